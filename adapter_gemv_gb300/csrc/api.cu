// api.cu -- the C ABI of libmlora (declared in include/mlora.h).
//
// Host side only: argument validation (every host-detectable error is returned before any
// launch), translation of the public structs into kernel parameter blocks, and dispatch to
// the kernels. Nothing here allocates device memory or synchronises the host.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "launch.h"
#include "mlora.h"

namespace {

thread_local char g_cuda_err[256] = "no CUDA error recorded";
std::atomic<int64_t> g_launches{0};
// lora_bgmv groups the rows of batches of at least this many rows on the device (bgmv_plan.cu).
constexpr int32_t kGroupDefaultMinRows = 128;
thread_local int g_pdl = 0;              // programmatic dependent launch for this thread's calls
thread_local uint64_t g_wait_limit_ns = 0;  // testing hook: 0 = the kernels' default limit

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int cuda_fail(cudaError_t e, const char *where) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return MLORA_ERR_CUDA;
}

// Checks a pool descriptor for the phases a call runs.
int check_pool(const mlora_pool *p, int32_t layer, bool need_a, bool need_b) {
  if (!p) return MLORA_ERR_NULL;
  if (p->dtype != MLORA_BF16 && p->dtype != MLORA_FP16) return MLORA_ERR_DTYPE;
  if (!p->rank || !p->scale) return MLORA_ERR_NULL;
  if (p->num_slots < 1 || p->num_layers < 1 || p->r_max < 1 || p->r_max > MLORA_MAX_RANK) return MLORA_ERR_SHAPE;
  if (p->d_in < 8 || p->d_out < 8) return MLORA_ERR_SHAPE;
  if (p->d_in % 8 || p->d_out % 8) return MLORA_ERR_ALIGN;
  if (layer < 0 || layer >= p->num_layers) return MLORA_ERR_SHAPE;
  if (!aligned(p->rank, 4) || !aligned(p->scale, 4)) return MLORA_ERR_ALIGN;
  if (p->kind == MLORA_POOL_STACKED) {
    if ((need_a && !p->a_t) || (need_b && !p->b)) return MLORA_ERR_NULL;
    if ((need_a && !aligned(p->a_t, 16)) || (need_b && !aligned(p->b, 16))) return MLORA_ERR_ALIGN;
  } else if (p->kind == MLORA_POOL_PAGED) {
    if (!p->pages || (need_a && !p->a_page_table) || (need_b && !p->b_page_table)) return MLORA_ERR_NULL;
    if (p->num_pages < 1 || p->page_elems < 8 || p->page_elems > INT32_MAX) return MLORA_ERR_POOL;
    if (p->num_pages > INT32_MAX) return MLORA_ERR_POOL;  // page ids are int32
    if (!aligned(p->pages, 16) || p->page_elems % 8) return MLORA_ERR_ALIGN;
    if ((need_a && !aligned(p->a_page_table, 4)) || (need_b && !aligned(p->b_page_table, 4))) return MLORA_ERR_ALIGN;
  } else {
    return MLORA_ERR_POOL;
  }
  return MLORA_OK;
}

mlora::PoolDev to_dev(const mlora_pool *p) {
  mlora::PoolDev d{};
  d.kind = p->kind;
  d.dtype = p->dtype;
  d.num_slots = p->num_slots;
  d.num_layers = p->num_layers;
  d.r_max = p->r_max;
  d.d_in = p->d_in;
  d.d_out = p->d_out;
  d.a_t = static_cast<const uint16_t *>(p->a_t);
  d.b = static_cast<const uint16_t *>(p->b);
  d.pages = static_cast<const uint16_t *>(p->pages);
  d.page_elems = p->page_elems;
  d.num_pages = p->num_pages;
  d.a_tab = p->a_page_table;
  d.b_tab = p->b_page_table;
  d.rank = p->rank;
  d.scale = p->scale;
  d.a_ppv = d.b_ppv = 1;
  d.pe_mul = 1;
  d.pe_shift = 0;
  if (p->kind == MLORA_POOL_PAGED) {  // a vector longer than a page spans several
    d.a_ppv = (int32_t)((p->d_in + p->page_elems - 1) / p->page_elems);
    d.b_ppv = (int32_t)((p->d_out + p->page_elems - 1) / p->page_elems);
    // division by page_elems as a multiply-high and a shift (Granlund and Montgomery, 1994)
    const uint64_t pe = (uint64_t)p->page_elems;
    int l = 0;
    while ((1ull << l) < pe) ++l;
    d.pe_mul = (uint32_t)(((1ull << 32) * ((1ull << l) - pe)) / pe + 1);
    d.pe_shift = l;
  }
  return d;
}

// With zero rows the activation, output and v pointers may be NULL (empty arrays).
int check_x(const void *x, int64_t ldx, const mlora_pool *p, int32_t rows) {
  if (rows == 0) return MLORA_OK;
  if (!x) return MLORA_ERR_NULL;
  if (ldx < p->d_in) return MLORA_ERR_SHAPE;
  if (!aligned(x, 16) || ldx % 8) return MLORA_ERR_ALIGN;
  return MLORA_OK;
}

int check_y(const void *y, int64_t ldy, const mlora_pool *p, int32_t rows) {
  if (rows == 0) return MLORA_OK;
  if (!y) return MLORA_ERR_NULL;
  if (ldy < p->d_out) return MLORA_ERR_SHAPE;
  if (!aligned(y, 16) || ldy % 8) return MLORA_ERR_ALIGN;
  return MLORA_OK;
}

int check_v(const float *v, int32_t rows) {
  if (rows == 0) return MLORA_OK;
  if (!v) return MLORA_ERR_NULL;
  if (!aligned(v, 4)) return MLORA_ERR_ALIGN;
  return MLORA_OK;
}

int check_rows_sgmv(const int32_t *off, const int32_t *slot, int32_t nseg, int32_t num_rows, const int32_t *status) {
  if (num_rows < 0 || nseg < 0) return MLORA_ERR_SHAPE;
  if (!off || (nseg > 0 && !slot)) return MLORA_ERR_NULL;
  if (!aligned(off, 4) || !aligned(slot, 4) || !aligned(status, 4)) return MLORA_ERR_ALIGN;
  return MLORA_OK;
}

int check_rows_bgmv(const int32_t *row_slot, int32_t num_rows, const int32_t *status) {
  if (num_rows < 0) return MLORA_ERR_SHAPE;
  if (num_rows > 0 && !row_slot) return MLORA_ERR_NULL;
  if (!aligned(row_slot, 4) || !aligned(status, 4)) return MLORA_ERR_ALIGN;
  return MLORA_OK;
}

#define TRY(expr)              \
  do {                         \
    const int rc_ = (expr);    \
    if (rc_ != MLORA_OK) return rc_; \
  } while (0)

mlora::DecodeParams base_params(const int32_t *off, const int32_t *seg_slot, int32_t nseg, const int32_t *row_slot,
                                int32_t num_rows, int32_t *status) {
  mlora::DecodeParams d{};
  d.seg_off = off;
  d.seg_slot = seg_slot;
  d.nseg = nseg;
  d.row_slot = row_slot;
  d.M = num_rows;
  d.status = status;
  return d;
}

int run(int mode, int dtype, mlora::DecodeParams d, void *stream, bool pdl) {
  d.wait_ns = g_wait_limit_ns;
  const cudaError_t e = mlora::launch_decode(mode, dtype, d, static_cast<cudaStream_t>(stream), pdl);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return MLORA_OK;
}

// The tensor-core kernels for the long segments of one problem (prefill_tc.cu): segments of at
// least tc_min_rows(nseg) rows, in blocks of at most 128 rows (the last one masked). Marks the
// problem so that the CUDA-core kernel launched after them takes only the shorter segments.
int run_tc(int mode, mlora::ProblemDev &q, const mlora_pool *pool, const int32_t *off, const int32_t *seg_slot,
           int32_t nseg, int32_t num_rows, int32_t *status, void *stream) {
  mlora::TcParams tp{};
  tp.num_slots = pool->num_slots;
  tp.num_layers = pool->num_layers;
  tp.r_max = pool->r_max;
  tp.d_in = pool->d_in;
  tp.d_out = pool->d_out;
  tp.layer = q.layer;
  tp.rank = pool->rank;
  tp.scale = pool->scale;
  tp.seg_off = off;
  tp.seg_slot = seg_slot;
  tp.nseg = nseg;
  tp.M = num_rows;
  tp.v = q.v;
  tp.y = q.y;
  tp.ldy = q.ldy;
  tp.status = status;
  tp.tc_min = mlora::tc_min_rows(nseg);
  tp.paged = q.pool.kind == MLORA_POOL_PAGED ? 1 : 0;
  tp.page_elems = (int32_t)q.pool.page_elems;
  tp.a_ppv = q.pool.a_ppv;
  tp.b_ppv = q.pool.b_ppv;
  tp.num_pages = q.pool.num_pages;
  tp.pages = q.pool.pages;
  tp.a_tab = q.pool.a_tab;
  tp.b_tab = q.pool.b_tab;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (mode != mlora::MODE_EXPAND) {
    const cudaError_t e = mlora::launch_tc_shrink(q, tp, st);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core shrink launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  if (mode != mlora::MODE_SHRINK) {
    const cudaError_t e = mlora::launch_tc_expand(q, tp, st, mode == mlora::MODE_FUSED);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core expand launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  q.tc_min = tp.tc_min;
  return MLORA_OK;
}

// A second stream, per host thread and device, for the CUDA-core launch of a call that also runs
// tensor-core kernels. The two take disjoint rows (the short and the long segments), so they may
// run at the same time: with a few long prompts mixed with decode rows the tensor-core kernels
// fill only part of the SMs, and the CUDA-core kernel's rows would otherwise wait behind them.
// Created on the thread's first such call whose stream is not being captured; until then (and
// for lora_sgmv_noalloc, which creates nothing) the launches stay on the caller's stream.
struct SideStream {
  cudaStream_t stream;
  cudaEvent_t forked, joined;  // caller's stream -> side stream, and back
  bool ready, failed;
};
thread_local SideStream g_side[mlora::kMaxDevices];

SideStream *side_stream(cudaStream_t caller) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= mlora::kMaxDevices) return nullptr;
  SideStream &s = g_side[dev];
  if (s.ready) return &s;
  if (s.failed) return nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(caller, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return nullptr;
  if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) {
    s.failed = true;
    return nullptr;
  }
  if (cudaEventCreateWithFlags(&s.forked, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&s.joined, cudaEventDisableTiming) != cudaSuccess) {
    s.failed = true;
    return nullptr;
  }
  s.ready = true;
  return &s;
}

// SGMV over the problems of d: for each problem whose batch may hold long segments (a prefill
// batch, or prefill and decode rows mixed), the tensor-core kernels take the segments of at least
// tc_min_rows(nseg) rows; one CUDA-core launch takes every other segment of every problem, on
// the side stream when there is one (forked from the caller's stream before the tensor-core
// launches, joined back after them).
int run_sgmv(int mode, mlora::DecodeParams &d, const mlora_pool *const *pools, void *stream, bool pdl,
             bool side_ok = true) {
  bool any_tc = false;
  for (int q = 0; q < d.nprob && !any_tc; ++q) any_tc = mlora::tc_eligible(d.prob[q].pool, d.M, d.nseg);
  if (!any_tc) return run(mode, pools[0]->dtype, d, stream, pdl);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SideStream *side = side_ok ? side_stream(st) : nullptr;
  if (side) {
    cudaError_t e = cudaEventRecord(side->forked, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->forked, 0);
    if (e != cudaSuccess) return cuda_fail(e, "fork to the side stream");
  }
  int rc = MLORA_OK;
  for (int q = 0; q < d.nprob && rc == MLORA_OK; ++q) {
    if (!mlora::tc_eligible(d.prob[q].pool, d.M, d.nseg)) continue;
    rc = run_tc(mode, d.prob[q], pools[q], d.seg_off, d.seg_slot, d.nseg, d.M, d.status, stream);
  }
  // after a tensor-core launch the CUDA-core kernel needs no early start (no PDL): on the caller's
  // stream its dependency is that launch; on the side stream, the work before the call. A fused
  // call on a pool of large ranks (the decode rows of a mixed batch, each on its own adapter)
  // streams its short segments instead (bgmv_stream.cu).
  if (rc == MLORA_OK) {
    cudaStream_t cst = side ? side->stream : st;
    if (mode == mlora::MODE_FUSED && d.nprob == 1 && d.nseg <= mlora::kStreamMaxSegs &&
        mlora::stream_eligible(d.prob[0].pool, d.M)) {
      const cudaError_t e = mlora::launch_sgmv_stream(d.prob[0], d.seg_off, d.seg_slot, d.nseg, d.prob[0].tc_min, d.M,
                                                      d.status, g_wait_limit_ns, cst);
      if (e != cudaSuccess) rc = cuda_fail(e, "streaming SGMV launch");
      else g_launches.fetch_add(1, std::memory_order_relaxed);
    } else {
      rc = run(mode, pools[0]->dtype, d, cst, false);
    }
  }
  if (side) {  // joined even after an error: nothing is left on the side stream (nor in a capture)
    cudaError_t e = cudaEventRecord(side->joined, side->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, side->joined, 0);
    if (e != cudaSuccess && rc == MLORA_OK) rc = cuda_fail(e, "join from the side stream");
  }
  return rc;
}

mlora::ProblemDev problem(const mlora_pool *pool, int32_t layer, const void *x, int64_t ldx, void *y, int64_t ldy,
                          float *v) {
  mlora::ProblemDev q{};
  q.pool = to_dev(pool);
  q.layer = layer;
  q.x = static_cast<const uint16_t *>(x);
  q.ldx = ldx;
  q.y = static_cast<uint16_t *>(y);
  q.ldy = ldy;
  q.v = v;
  return q;
}

// Built-in scratch of lora_sgmv_noalloc: the v rows of one call (num_rows x r_max floats).
// In host code the name is only a stand-in for the symbol; the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) float g_noalloc_v[MLORA_NOALLOC_MAX_FLOATS];
std::mutex g_noalloc_mu;
float *g_noalloc_ptr[256] = {};  // device address per device ordinal

int noalloc_scratch(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 256) return MLORA_ERR_SHAPE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_v);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch");
    g_noalloc_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MLORA_OK;
}

}  // namespace

extern "C" {

int lora_sgmv_shrink(float *v, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *seg_offsets,
                     const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t layer,
                     int32_t *dev_status, void *stream) {
  TRY(check_pool(pool, layer, true, false));
  TRY(check_v(v, num_rows));
  TRY(check_x(x, ldx, pool, num_rows));
  TRY(check_rows_sgmv(seg_offsets, seg_slot, num_segments, num_rows, dev_status));
  if (num_rows == 0) return MLORA_OK;
  mlora::DecodeParams d = base_params(seg_offsets, seg_slot, num_segments, nullptr, num_rows, dev_status);
  d.prob[0] = problem(pool, layer, x, ldx, nullptr, 0, v);
  d.nprob = 1;
  return run_sgmv(mlora::MODE_SHRINK, d, &pool, stream, g_pdl != 0);
}

int lora_sgmv_expand(void *y, int64_t ldy, const float *v, const mlora_pool *pool, const int32_t *seg_offsets,
                     const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t layer,
                     int32_t *dev_status, void *stream) {
  TRY(check_pool(pool, layer, false, true));
  TRY(check_v(v, num_rows));
  TRY(check_y(y, ldy, pool, num_rows));
  TRY(check_rows_sgmv(seg_offsets, seg_slot, num_segments, num_rows, dev_status));
  if (num_rows == 0) return MLORA_OK;
  mlora::DecodeParams d = base_params(seg_offsets, seg_slot, num_segments, nullptr, num_rows, dev_status);
  d.prob[0] = problem(pool, layer, nullptr, 0, y, ldy, const_cast<float *>(v));
  d.nprob = 1;
  return run_sgmv(mlora::MODE_EXPAND, d, &pool, stream, g_pdl != 0);
}

int lora_bgmv_shrink(float *v, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *row_slot,
                     int32_t num_rows, int32_t layer, int32_t *dev_status, void *stream) {
  TRY(check_pool(pool, layer, true, false));
  TRY(check_v(v, num_rows));
  TRY(check_x(x, ldx, pool, num_rows));
  TRY(check_rows_bgmv(row_slot, num_rows, dev_status));
  if (num_rows == 0) return MLORA_OK;
  mlora::DecodeParams d = base_params(nullptr, nullptr, 0, row_slot, num_rows, dev_status);
  d.prob[0] = problem(pool, layer, x, ldx, nullptr, 0, v);
  d.nprob = 1;
  return run(mlora::MODE_SHRINK, pool->dtype, d, stream, g_pdl != 0);
}

int lora_bgmv_expand(void *y, int64_t ldy, const float *v, const mlora_pool *pool, const int32_t *row_slot,
                     int32_t num_rows, int32_t layer, int32_t *dev_status, void *stream) {
  TRY(check_pool(pool, layer, false, true));
  TRY(check_v(v, num_rows));
  TRY(check_y(y, ldy, pool, num_rows));
  TRY(check_rows_bgmv(row_slot, num_rows, dev_status));
  if (num_rows == 0) return MLORA_OK;
  mlora::DecodeParams d = base_params(nullptr, nullptr, 0, row_slot, num_rows, dev_status);
  d.prob[0] = problem(pool, layer, nullptr, 0, y, ldy, const_cast<float *>(v));
  d.nprob = 1;
  return run(mlora::MODE_EXPAND, pool->dtype, d, stream, g_pdl != 0);
}

int lora_sgmv(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *seg_offsets,
              const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t layer, float *v_scratch,
              int32_t *dev_status, void *stream) {
  TRY(check_pool(pool, layer, true, true));
  TRY(check_v(v_scratch, num_rows));
  TRY(check_x(x, ldx, pool, num_rows));
  TRY(check_y(y, ldy, pool, num_rows));
  TRY(check_rows_sgmv(seg_offsets, seg_slot, num_segments, num_rows, dev_status));
  if (num_rows == 0) return MLORA_OK;
  mlora::DecodeParams d = base_params(seg_offsets, seg_slot, num_segments, nullptr, num_rows, dev_status);
  d.prob[0] = problem(pool, layer, x, ldx, y, ldy, v_scratch);
  d.nprob = 1;
  return run_sgmv(mlora::MODE_FUSED, d, &pool, stream, g_pdl != 0);
}

int lora_sgmv_noalloc(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool,
                      const int32_t *seg_offsets, const int32_t *seg_slot, int32_t num_segments, int32_t num_rows,
                      int32_t layer, int32_t *dev_status, void *stream) {
  TRY(check_pool(pool, layer, true, true));
  TRY(check_x(x, ldx, pool, num_rows));
  TRY(check_y(y, ldy, pool, num_rows));
  TRY(check_rows_sgmv(seg_offsets, seg_slot, num_segments, num_rows, dev_status));
  if ((int64_t)num_rows * pool->r_max > MLORA_NOALLOC_MAX_FLOATS) return MLORA_ERR_TOO_LARGE;
  if (num_rows == 0) return MLORA_OK;
  float *v = nullptr;
  TRY(noalloc_scratch(&v));
  mlora::DecodeParams d = base_params(seg_offsets, seg_slot, num_segments, nullptr, num_rows, dev_status);
  d.prob[0] = problem(pool, layer, x, ldx, y, ldy, v);
  d.nprob = 1;
  return run_sgmv(mlora::MODE_FUSED, d, &pool, stream, g_pdl != 0, false);
}

int lora_bgmv_ex(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *row_slot,
                 int32_t num_rows, int32_t layer, float *v_scratch, uint32_t flags, int32_t *dev_status,
                 void *stream) {
  if (flags & ~(MLORA_LAUNCH_PROGRAMMATIC | MLORA_LAUNCH_GROUP_ROWS | MLORA_LAUNCH_NO_GROUPING)) return MLORA_ERR_SHAPE;
  TRY(check_pool(pool, layer, true, true));
  TRY(check_v(v_scratch, num_rows));
  TRY(check_x(x, ldx, pool, num_rows));
  TRY(check_y(y, ldy, pool, num_rows));
  TRY(check_rows_bgmv(row_slot, num_rows, dev_status));
  if (num_rows == 0) return MLORA_OK;
  const bool pdl = (flags & MLORA_LAUNCH_PROGRAMMATIC) != 0;
  mlora::DecodeParams d = base_params(nullptr, nullptr, 0, row_slot, num_rows, dev_status);
  d.prob[0] = problem(pool, layer, x, ldx, y, ldy, v_scratch);
  d.nprob = 1;
  // Grouping: requested, or by default for batches large enough for repeated adapters to matter.
  // The order goes to v_scratch (two int32 per row), which the fused kernel does not use.
  const bool want = (flags & MLORA_LAUNCH_GROUP_ROWS) != 0 ||
                    ((flags & MLORA_LAUNCH_NO_GROUPING) == 0 && num_rows >= kGroupDefaultMinRows);
  if (want && num_rows <= mlora::kPlanMaxRows && pool->r_max >= 2) {
    int32_t *perm = reinterpret_cast<int32_t *>(v_scratch);
    int32_t *sslot = perm + num_rows;
    // heterogeneous ranks: the grouped order is cut into segments of rows that share a slot
    // (after perm and sslot in v_scratch: num_rows + 1 more int32), which the streaming kernel
    // takes a cluster of CTAs at a time
    const bool stream_rows = mlora::stream_eligible(d.prob[0].pool, num_rows);
    int32_t *segs = stream_rows ? sslot + num_rows : nullptr;
    const cudaError_t e = mlora::launch_bgmv_plan(row_slot, num_rows, d.prob[0].pool, perm, sslot, segs,
                                                  mlora::kStreamSegRows, static_cast<cudaStream_t>(stream), pdl);
    if (e != cudaSuccess) return cuda_fail(e, "row grouping launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (stream_rows) {  // reads the order: no early start
      const cudaError_t es = mlora::launch_bgmv_stream(d.prob[0], perm, sslot, segs, num_rows, dev_status,
                                                       g_wait_limit_ns, static_cast<cudaStream_t>(stream));
      if (es != cudaSuccess) return cuda_fail(es, "streaming BGMV launch");
      g_launches.fetch_add(1, std::memory_order_relaxed);
      return MLORA_OK;
    }
    d.perm = perm;
    d.sslot = sslot;
    return run(mlora::MODE_FUSED, pool->dtype, d, stream, false);  // reads the order: no early start
  }
  return run(mlora::MODE_FUSED, pool->dtype, d, stream, pdl);
}

int lora_bgmv(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *row_slot,
              int32_t num_rows, int32_t layer, float *v_scratch, int32_t *dev_status, void *stream) {
  return lora_bgmv_ex(y, ldy, x, ldx, pool, row_slot, num_rows, layer, v_scratch,
                      g_pdl ? MLORA_LAUNCH_PROGRAMMATIC : 0u, dev_status, stream);
}

}  // extern "C"

namespace {

// Validates one grouped call and fills its parameter block (no launch).
int prepare_grouped(const mlora_problem *problems, int32_t num_problems, const int32_t *seg_offsets,
                    const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t *dev_status,
                    mlora::DecodeParams &d, const mlora_pool **pools) {
  if (!problems) return MLORA_ERR_NULL;
  if (num_problems < 1 || num_problems > MLORA_MAX_GROUP) return MLORA_ERR_SHAPE;
  TRY(check_rows_sgmv(seg_offsets, seg_slot, num_segments, num_rows, dev_status));
  d = base_params(seg_offsets, seg_slot, num_segments, nullptr, num_rows, dev_status);
  for (int q = 0; q < num_problems; ++q) {
    const mlora_problem &pb = problems[q];
    TRY(check_pool(pb.pool, pb.layer, true, true));
    if (pb.pool->dtype != problems[0].pool->dtype) return MLORA_ERR_DTYPE;
    TRY(check_v(pb.v_scratch, num_rows));
    TRY(check_x(pb.x, pb.ldx, pb.pool, num_rows));
    TRY(check_y(pb.y, pb.ldy, pb.pool, num_rows));
    d.prob[q] = problem(pb.pool, pb.layer, pb.x, pb.ldx, pb.y, pb.ldy, pb.v_scratch);
    pools[q] = pb.pool;
  }
  d.nprob = num_problems;
  return MLORA_OK;
}

}  // namespace

extern "C" {

int lora_sgmv_grouped_ex(const mlora_problem *problems, int32_t num_problems, const int32_t *seg_offsets,
                         const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, uint32_t flags,
                         int32_t *dev_status, void *stream) {
  if (flags & ~MLORA_LAUNCH_PROGRAMMATIC) return MLORA_ERR_SHAPE;
  mlora::DecodeParams d;
  const mlora_pool *pools[MLORA_MAX_GROUP];
  TRY(prepare_grouped(problems, num_problems, seg_offsets, seg_slot, num_segments, num_rows, dev_status, d, pools));
  if (num_rows == 0) return MLORA_OK;
  return run_sgmv(mlora::MODE_FUSED, d, pools, stream, (flags & MLORA_LAUNCH_PROGRAMMATIC) != 0);
}

int lora_sgmv_sequence(const mlora_group *groups, int32_t num_groups, uint32_t flags, int32_t *dev_status,
                       void *stream) {
  if (!groups) return MLORA_ERR_NULL;
  if (num_groups < 0) return MLORA_ERR_SHAPE;
  if (flags & ~MLORA_LAUNCH_PROGRAMMATIC) return MLORA_ERR_SHAPE;
  struct Prepared {
    mlora::DecodeParams d;
    const mlora_pool *pools[MLORA_MAX_GROUP];
  };
  std::vector<Prepared> calls((size_t)num_groups);
  for (int g = 0; g < num_groups; ++g) {
    const mlora_group &gr = groups[g];
    TRY(prepare_grouped(gr.problems, gr.num_problems, gr.seg_offsets, gr.seg_slot, gr.num_segments, gr.num_rows,
                        dev_status, calls[g].d, calls[g].pools));
  }
  bool first = true;
  for (int g = 0; g < num_groups; ++g) {
    if (groups[g].num_rows == 0) continue;
    const bool pdl = (flags & MLORA_LAUNCH_PROGRAMMATIC) != 0 && !first;
    TRY(run_sgmv(mlora::MODE_FUSED, calls[g].d, calls[g].pools, stream, pdl));
    first = false;
  }
  return MLORA_OK;
}

int lora_sgmv_grouped(const mlora_problem *problems, int32_t num_problems, const int32_t *seg_offsets,
                      const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t *dev_status,
                      void *stream) {
  return lora_sgmv_grouped_ex(problems, num_problems, seg_offsets, seg_slot, num_segments, num_rows,
                              g_pdl ? MLORA_LAUNCH_PROGRAMMATIC : 0u, dev_status, stream);
}

const char *lora_error_string(int code) {
  switch (code) {
    case MLORA_OK: return "ok";
    case MLORA_ERR_NULL: return "a required pointer is NULL";
    case MLORA_ERR_DTYPE: return "unsupported or mismatched dtype";
    case MLORA_ERR_SHAPE: return "a size or index is out of range";
    case MLORA_ERR_ALIGN: return "alignment rule broken (16-byte pointers, multiples of 8 elements)";
    case MLORA_ERR_POOL: return "malformed adapter pool descriptor";
    case MLORA_ERR_CUDA: return g_cuda_err;
    case MLORA_ERR_TOO_LARGE: return "num_rows * r_max exceeds the built-in scratch (MLORA_NOALLOC_MAX_FLOATS)";
    default: return "unknown error code";
  }
}

int lora_abi_version(void) { return MLORA_ABI_VERSION; }

int lora_set_programmatic_launch(int enable) {
  const int prev = g_pdl;
  g_pdl = enable ? 1 : 0;
  return prev;
}

void lora_test_set_wait_limit_ns(uint64_t limit_ns) { g_wait_limit_ns = limit_ns; }

int64_t lora_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
