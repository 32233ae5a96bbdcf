// launch.h -- parameter blocks and launchers shared by the C ABI and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mlora.h"

namespace mlora {

struct PoolDev {
  int32_t kind, dtype, num_slots, num_layers, r_max, d_in, d_out;
  const uint16_t *a_t, *b, *pages;
  int64_t page_elems, num_pages;
  const int32_t *a_tab, *b_tab, *rank;  // paged: [slot][layer][r_max][a_ppv or b_ppv] page ids
  const float *scale;
  int32_t a_ppv, b_ppv;  // paged: pages per vector, ceil(d_in / page_elems), ceil(d_out / page_elems)
  uint32_t pe_mul;       // paged: k / page_elems = (mulhi(pe_mul, k) + k) >> pe_shift for k < 2^31
  int32_t pe_shift;
};

enum { MODE_SHRINK = 0, MODE_EXPAND = 1, MODE_FUSED = 2 };

// One projection of a launch.
struct ProblemDev {
  PoolDev pool;
  int32_t layer;
  const uint16_t *x;
  int64_t ldx;
  uint16_t *y;
  int64_t ldy;
  float *v;  // [M][r_max]
  int32_t tc_min;  // > 0: segments of at least tc_min rows are done by the tensor-core kernels;
                   // the CUDA-core kernel takes only the shorter segments of this problem
};

struct DecodeParams {
  ProblemDev prob[MLORA_MAX_GROUP];
  int32_t nprob;
  const int32_t *seg_off, *seg_slot;  // SGMV (seg_off != nullptr)
  int32_t nseg;
  const int32_t *row_slot;  // BGMV
  const int32_t *perm, *sslot;  // BGMV in grouped order (bgmv_plan.cu): tile t is row perm[t], slot sslot[t]
  int32_t M;
  int32_t *status;
  uint64_t wait_ns;  // limit of the kernel's waits (0 = the default, kWaitLimitNs)
  // chosen by the launcher
  int32_t npt;  // paged pools: page-table entries of a tile kept in shared memory (0: none)
  int32_t rt, tiles, csplit, kb, nb, ny, xw, r_alloc;  // nb: staged B columns; ny: y slice staged;
                                                      // xw: x row width staged (whole d_in slice), 0 = one pass
};

// Tensor-core path for the full 128-row blocks of long SGMV segments (prefill_tc.cu).
struct TcParams {
  int32_t num_slots, num_layers, r_max, d_in, d_out, layer;
  const int32_t *rank;
  const float *scale;
  const int32_t *seg_off, *seg_slot;
  int32_t nseg, M;
  float *v;  // [M][r_max] fp32: written by the shrink, read by the expand
  uint16_t *y;
  int64_t ldy;
  int32_t *status;
  int32_t tc_min;  // segments of at least this many rows are this path's
  // chosen by the launcher
  int32_t rpad, ksplit, tiles, nper, nblk_total, tmem_cols, stages;
  int32_t bm;  // rows per tile (a multiple of 8, at most the MMA's 128)
  // paged pools: the A^T / B tiles are gathered row by row from the pages
  int32_t paged, page_elems, a_ppv, b_ppv;
  int64_t num_pages;
  const uint16_t *pages;
  const int32_t *a_tab, *b_tab;
};

// Segments of at least tc_min rows go to the tensor-core kernels, the shorter ones to the CUDA-core
// kernel, whose launch is sized for the worst case the host can see: every segment just short of
// tc_min rows. The host picks tc_min per call (tc_min_rows): kTcMinRows, lowered towards
// kTcMinRowsLow so that this worst case stays near one CTA per SM -- in a prefill batch of a few long
// prompts that launch is otherwise mostly empty tiles (8 prompts, 13B fused call: 18 us of a 115 us
// call).
constexpr int kTcMinRows = 32;
constexpr int kTcMinRowsLow = 8;
int tc_min_rows(int nseg);

// Number of SMs of the current device (cached per device ordinal, safe from any host thread).
int sm_count();
constexpr int kMaxDevices = 64;  // devices with a cached entry; others are queried on every call

// Whether an SGMV call over num_rows rows in nseg segments on this pool launches the tensor-core
// kernels for its long segments (decided on the host, which does not see the segment lengths).
bool tc_eligible(const PoolDev &pool, int num_rows, int nseg);
cudaError_t launch_tc_shrink(const ProblemDev &pr, TcParams p, cudaStream_t stream);
// after_shrink: launched right behind launch_tc_shrink of the same problem on the same stream
// (a fused call); the expand then starts early and waits for the shrink before reading v.
cudaError_t launch_tc_expand(const ProblemDev &pr, TcParams p, cudaStream_t stream, bool after_shrink);

// Device-side grouping of BGMV rows (bgmv_plan.cu): the rows in order of (rank descending, slot,
// row) into perm / sslot [num_rows] each. At most kPlanMaxRows rows.
// With segs != nullptr the order is also cut into segments of at most seg_rows rows that share a
// slot: segs[0] = the count, segs[1 + k] = segment k's first position (M + 1 int32 at most).
constexpr int kPlanMaxRows = 4096;
cudaError_t launch_bgmv_plan(const int32_t *row_slot, int32_t M, const PoolDev &pool, int32_t *perm, int32_t *sslot,
                             int32_t *segs, int32_t seg_rows, cudaStream_t stream, bool pdl);

// BGMV rows of a heterogeneous-rank pool, in the grouped order cut into segments of rows that share
// a slot: a cluster of CTAs per segment streams the adapter's A^T and B rank-rows through
// shared-memory rings (bgmv_stream.cu).
constexpr int kStreamSegRows = 4;  // rows per segment at most
struct StreamParams {
  ProblemDev pr;
  const int32_t *perm, *sslot;  // BGMV: the grouped order (bgmv_plan.cu)
  const int32_t *segs;          // BGMV: [0] segment count, [1 + k] first position of segment k
  // SGMV (seg_off != nullptr): the call's segments; those shorter than tc_min rows are this
  // kernel's (the longer ones go to the tensor-core kernels), cut into pieces of kStreamSegRows
  const int32_t *seg_off, *seg_slot;
  int32_t nseg, tc_min;
  int32_t M;
  int32_t *status;
  uint64_t wait_ns;
  int32_t cs, kc, nc;    // CTAs per segment (a cluster), each CTA's slice of d_in and of d_out
  int32_t kpad, stages;  // x slice buffer width (elements), ring stages
  int32_t ptn;           // paged pools: page-table entries of one slot (r_max (a_ppv + b_ppv))
};
// Whether lora_bgmv's grouped rows on this pool take the streaming kernel (r_max of 32 to 128 and
// the buffers fit in shared memory).
bool stream_eligible(const PoolDev &pool, int num_rows);
cudaError_t launch_bgmv_stream(const ProblemDev &pr, const int32_t *perm, const int32_t *sslot, const int32_t *segs,
                               int32_t M, int32_t *status, uint64_t wait_ns, cudaStream_t stream);
// The short segments of an SGMV call whose long segments the tensor-core kernels take (at most
// kStreamMaxSegs segments).
constexpr int kStreamMaxSegs = 1024;
cudaError_t launch_sgmv_stream(const ProblemDev &pr, const int32_t *seg_off, const int32_t *seg_slot, int32_t nseg,
                               int32_t tc_min, int32_t M, int32_t *status, uint64_t wait_ns, cudaStream_t stream);

// CUDA-core path for decode-sized tiles (decode_launch.cu chooses the split and the stages;
// decode_{shrink,expand,fused}.cu hold the kernels). force_csplit > 0 overrides the split.
cudaError_t launch_decode(int mode, int dtype, DecodeParams p, cudaStream_t stream, bool pdl, int force_csplit = 0);

cudaError_t launch_decode_shrink(int dtype, const DecodeParams &p, unsigned grid, size_t smem, int cluster, bool pdl,
                                 cudaStream_t stream);
cudaError_t launch_decode_expand(int dtype, const DecodeParams &p, unsigned grid, size_t smem, int cluster, bool pdl,
                                 cudaStream_t stream);
cudaError_t launch_decode_fused(int dtype, const DecodeParams &p, unsigned grid, size_t smem, int cluster, bool pdl,
                                cudaStream_t stream);

}  // namespace mlora
