// bgmv_stream.cu -- BGMV rows of a heterogeneous-rank pool streamed through shared-memory rings
// (sm_103a, CUDA cores).
//
// S-LoRA serves thousands of adapters of different ranks from one paged pool and batches their
// decode rows together (S-LoRA section 3, "Heterogeneous Batching Kernels" and "Unified
// Paging"): a rank-64 row moves eight times the bytes of a rank-8 row, and popular adapters
// serve many rows of one batch. The device-side grouping (bgmv_plan.cu) orders the rows by rank,
// largest first, then by slot, and cuts the order into segments of at most RSEG rows that share a
// slot (Punica section 3.4, "Batch Layout Construction": rows of one adapter form one group). This
// kernel gives each segment to a cluster of cs CTAs. CTA c of the cluster streams its slice c of
// d_in of the adapter's A^T rank-rows, then its slice c of d_out of the B rank-rows, once for all
// the segment's rows, through a ring of shared-memory stages filled by bulk copies, so every CTA
// keeps up to 128 KB in flight whatever the rank and never reloads operands from L2 after a wait:
//   * one producer warp per CTA resolves each segment (slot, rank, scale, page ids, checked; the
//     rows), publishes it in a descriptor and issues the bulk copies: the slices of the segment's x
//     rows, then the stages -- a stage is 64 KB: A^T's groups of 8 rank-rows x 4096 elements for
//     every chunk of the d_in slice, then B's groups of 16 rank-rows x 2048 columns for every chunk
//     of the d_out slice (a stage's handoff costs about as much for 32 KB as for 64 KB);
//   * eight consumer warps: for an A stage, warp w dots its two 256-element slices of each of the
//     stage's 8 rank-rows with every row's x slice, held in registers (mixed-precision FMAs, one
//     fp32 chain per rank-row and row), and after the group's last chunk sums the chains over its
//     lanes into shared memory; the warps' sums are added in warp order once per segment (Punica
//     section 3.4, the shrink, split over d_in); the cluster's partial
//     sums are pushed into every peer's shared memory (st.async, completing on the receiver's
//     mbarrier) and summed in CTA-rank order; for a B stage, thread t accumulates its 8 columns of
//     every row over the group's rank-rows (paired fp32 FMAs) and, after the chunk's last group,
//     writes y = rn(y + scale * sum) (the expand, split over d_out);
//   * the stages cycle through full / empty mbarriers. Every wait is bounded: a CTA that gives up
//     reports MLORA_STATUS_TIMEOUT, stops issuing and, before it exits, waits (bounded) for the
//     copies it issued and the partial sums its peers may still push.
// The persistent grid of clusters takes the segments in snake order (cluster b gets segments b,
// 2C - 1 - b, 2C + b, ... of C clusters), which balances their sizes, largest first. Rows without
// adapter are skipped (y untouched); invalid slots, ranks and page ids are reported and their rows
// skipped. The sums run in a fixed order (a call is deterministic); it is another order than the
// decode kernel's, within the same tolerance.
#include <cuda_runtime.h>

#include <type_traits>

#include "decode_impl.cuh"
#include "launch.h"

namespace mlora {
namespace bstream {

constexpr int CWARPS = 8;                    // consumer warps
constexpr int NTHREADS = (CWARPS + 1) * 32;  // + the producer warp
constexpr int ROWS = 8;                      // A^T stages: rank-rows per stage
constexpr int ACHUNK = 4096;                 //             elements of each rank-row per stage
constexpr int BROWS = 16;                    // B stages: rank-rows per stage
constexpr int CHUNK = 2048;                  //           columns of each rank-row per stage
constexpr int STAGE_BYTES = ROWS * ACHUNK * 2;  // 64 KB: the handoffs of a stage cost as much for 32 KB
static_assert(BROWS * CHUNK == ROWS * ACHUNK, "A^T and B stages of one size");
constexpr int RQ = 2;                        // segments in flight (descriptors, exchange buffers)
constexpr int MAX_STAGES = 8;
constexpr int MAX_RANK = 128;
constexpr int MAX_CS = 2;                    // CTAs per segment (cluster)
constexpr int MAX_PT = 2048;                 // page-table entries of one slot kept in shared memory

struct SegDesc {
  int32_t nrows, rank, bad, pad;
  float scale;
  int32_t rows[kStreamSegRows];  // the segment's rows (batch row indices)
};
constexpr int RSEG = kStreamSegRows;

// Shared memory:
//   [0, 512)         barriers
//   [512, 1024)      RQ segment descriptors and the stop flag
//   vx               [RQ][MAX_CS][RSEG][MAX_RANK] fp32: partial v of every CTA of the cluster
//   vsm              [RSEG][MAX_RANK] fp32: the summed v
//   red              [gmax][CWARPS][32] fp32: the consumer warps' lane sums of every rank-row group
//                    of the segment (gmax = r_max / 8 rounded up)
//   pt               [RQ][ptn] int32: page ids of the segments in flight (paged pools: the producer
//                    reads a slot's page-table entries once, when it checks them)
//   x                [RSEG][kpad]: the x slices of the segment's rows (one segment at a time)
//   ring             [stages][32 KB]
//   (SGMV: [1024, 5124) the first unit of every segment of the call, and the unit count)
struct Smem {
  int vx, vsm, red, pt, x, ring, total;
  __host__ __device__ static Smem make(int kpad, int ptn, int stages, int gmax) {
    Smem s;
    s.vx = 1024 + (kStreamMaxSegs + 1) * 4;
    s.vsm = s.vx + RQ * MAX_CS * RSEG * MAX_RANK * 4;
    s.red = s.vsm + RSEG * MAX_RANK * 4;
    s.pt = s.red + gmax * CWARPS * 32 * 4;
    s.x = (s.pt + RQ * ptn * 4 + 127) & ~127;
    s.ring = (s.x + RSEG * kpad * 2 + 1023) & ~1023;
    s.total = s.ring + stages * STAGE_BYTES;
    return s;
  }
};

// OR of v over the consumer warps (named barrier 1): every consumer thread gets the same answer,
// so they leave their loops together.
__device__ __forceinline__ int consumers_or(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, 1, %2, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v), "n"(CWARPS * 32)
      : "memory");
  return r;
}

// One arrival on the mbarrier at shared::cluster address `remote` (a peer CTA's).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Eight products of chunk xv with chunk av (8 packed 16-bit elements each) into one fp32 chain,
// mixed-precision FMAs (16-bit operands, fp32 accumulator, one rounding per product).
template <int DT>
__device__ __forceinline__ void mfma8_chain(const uint4 &xv, const uint4 &av, float &c) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, as[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if constexpr (DT == MLORA_BF16)
      asm("{ .reg .b16 xl, xh, al, ah; mov.b32 {xl, xh}, %1; mov.b32 {al, ah}, %2;\n"
          " fma.rn.f32.bf16 %0, xl, al, %0; fma.rn.f32.bf16 %0, xh, ah, %0; }"
          : "+f"(c) : "r"(xs[q]), "r"(as[q]));
    else
      asm("{ .reg .b16 xl, xh, al, ah; mov.b32 {xl, xh}, %1; mov.b32 {al, ah}, %2;\n"
          " fma.rn.f32.f16 %0, xl, al, %0; fma.rn.f32.f16 %0, xh, ah, %0; }"
          : "+f"(c) : "r"(xs[q]), "r"(as[q]));
  }
}

// Sums of N values (N = 8, 16 or 32) over the 32 lanes of a warp, scattered over the lanes: each
// butterfly step halves the values a lane keeps (the lanes with the step's bit set keep the upper
// half and send the lower), so after the halving steps lane l holds the sum of value l / (32 / N)
// (the remaining steps add across the lanes that share it). 31 shuffles for N = 32, against
// 160 for a full reduction of every value.
template <int N>
__device__ __forceinline__ float lane_sum_scatter(float (&v)[N], int lane) {
  constexpr int H = N == 32 ? 5 : N == 16 ? 4 : 3;
  static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 values");
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int sft = 16 >> st;
    if (st < H) {
      const int n = N >> st;
      const bool up = (lane & sft) != 0;
#pragma unroll
      for (int k = 0; k < n / 2; ++k) {
        const float send = up ? v[k] : v[k + n / 2];
        const float keep = up ? v[k + n / 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], sft);
    }
  }
  return v[0];
}

// Unit i of cluster b of C in snake order.
__device__ __forceinline__ int snake(int i, int b, int C) { return i * C + ((i & 1) ? C - 1 - b : b); }

template <int DT>
__global__ void __launch_bounds__(NTHREADS, 1) stream_kernel(const __grid_constant__ StreamParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [MAX_STAGES]
  uint64_t *empty = full + MAX_STAGES;                   // [MAX_STAGES]
  uint64_t *segfull = empty + MAX_STAGES;                // [RQ]
  uint64_t *segempty = segfull + RQ;                     // [RQ]
  uint64_t *vfull = segempty + RQ;                       // [RQ] the peers' partial sums landed
  uint64_t *vempty = vfull + RQ;                         // [RQ] the peers consumed this CTA's partial sums
  uint64_t *xfull = vempty + RQ;                         // the x slices landed
  uint64_t *xempty = xfull + 1;                          // the consumers are done with the x slices
  SegDesc *desc = reinterpret_cast<SegDesc *>(smem + 512);
  volatile int32_t *stop = reinterpret_cast<volatile int32_t *>(smem + 512 + RQ * sizeof(SegDesc));
  const Smem S = Smem::make(p.kpad, p.ptn, p.stages, (p.pr.pool.r_max + ROWS - 1) / ROWS);
  float *vx = reinterpret_cast<float *>(smem + S.vx);
  float *vsm = reinterpret_cast<float *>(smem + S.vsm);
  uint16_t *xbuf = reinterpret_cast<uint16_t *>(smem + S.x);
  uint8_t *ring = smem + S.ring;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const ProblemDev &pr = p.pr;
  const PoolDev &pl = pr.pool;
  const int cs = p.cs, NS = p.stages;
  const int c = cs > 1 ? (int)cluster_ctarank() : 0;
  const int cb = (int)blockIdx.x / cs, C = (int)gridDim.x / cs;  // this cluster, the clusters
  int32_t *ufirst = reinterpret_cast<int32_t *>(smem + 1024);     // SGMV: [nseg + 1]
  // this CTA's slices of d_in and d_out
  const int k0 = min(c * p.kc, pl.d_in), k1 = min(k0 + p.kc, pl.d_in);
  const int n0 = min(c * p.nc, pl.d_out), n1 = min(n0 + p.nc, pl.d_out);
  const int kchunks = (k1 - k0 + ACHUNK - 1) / ACHUNK, nchunks = (n1 - n0 + CHUNK - 1) / CHUNK;
  const uint64_t wlim = p.wait_ns ? p.wait_ns : kWaitLimitNs;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CWARPS);
    }
    for (int q = 0; q < RQ; ++q) {
      mbar_init(&segfull[q], 1);
      mbar_init(&segempty[q], CWARPS);
      mbar_init(&vfull[q], 1);
      mbar_init(&vempty[q], cs > 1 ? cs - 1 : 1);
    }
    mbar_init(xfull, 1);
    mbar_init(xempty, CWARPS);
    *stop = 0;
    mbar_fence_init();
  }
  // The units of work: BGMV, the plan kernel's segments; SGMV, the pieces of at most RSEG rows of
  // the segments shorter than tc_min (warp 0 counts them and checks the offsets, as the decode
  // kernel does: a malformed list is reported and nothing is done).
  if (p.seg_off != nullptr && warp == 0) {
    const int per = (p.nseg + 32) / 32;  // segments per lane, (nseg + 1) entries in all
    int32_t cnt = 0, bad = 0;
    for (int q = lane * per; q < min((lane + 1) * per, p.nseg); ++q) {
      const int32_t a = p.seg_off[q], b = p.seg_off[q + 1], len = b - a;
      bad |= (len < 0) | (a < 0) | (b > p.M);
      cnt += (len > 0 && len < p.tc_min) ? (len + RSEG - 1) / RSEG : 0;
    }
    if (lane == 0) bad |= p.nseg > 0 ? (p.seg_off[0] != 0) | (p.seg_off[p.nseg] != p.M) : (p.M != 0);
    int32_t incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int32_t run = incl - cnt;
    for (int q = lane * per; q < min((lane + 1) * per, p.nseg); ++q) {
      ufirst[q] = run;
      const int32_t len = p.seg_off[q + 1] - p.seg_off[q];
      run += (len > 0 && len < p.tc_min) ? (len + RSEG - 1) / RSEG : 0;
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 31) ufirst[p.nseg] = bad ? 0 : incl;
    if (bad && lane == 0 && blockIdx.x == 0) report(p.status, MLORA_STATUS_BAD_OFFSETS);
  }
  __syncthreads();
  const int nseg = p.seg_off != nullptr ? ufirst[p.nseg] : p.segs[0];  // units
  // x past the slice is zero (the copies write [0, k1 - k0) of each row only): a chunk's tail then
  // adds nothing, whatever stale bytes its stage holds (those are masked on the A side too)
  for (int e = (k1 - k0) + tid * 8; e < p.kpad; e += NTHREADS * 8)
    for (int r = 0; r < RSEG; ++r) *reinterpret_cast<uint4 *>(xbuf + r * p.kpad + e) = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (cs > 1) cluster_sync();  // every peer's barriers are initialised before anything is pushed

  if (warp == CWARPS) {
    // ------------------------------------------------------------------ producer warp
    const uint64_t pol = policy_evict_first();
    uint32_t ctr = 0;   // stages issued
    uint32_t xuse = 0;  // x copies issued (valid segments)
    bool ok = true;
    for (int i = 0;; ++i) {
      const int sg = snake(i, cb, C);
      if (sg >= nseg) break;
      const int q = i % RQ;
      const uint32_t use = (uint32_t)(i / RQ);
      ok = __all_sync(0xffffffffu, (use == 0 || mbar_wait(&segempty[q], (use - 1) & 1u, wlim)) && !*stop);
      if (!ok) break;
      int t0, t1, s;
      if (p.seg_off != nullptr) {  // the segment holding unit sg (the last whose first unit is <= sg) and its piece
        int lo = 0, hi = p.nseg;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (ufirst[mid] <= sg) lo = mid;
          else hi = mid;
        }
        t0 = p.seg_off[lo] + (sg - ufirst[lo]) * RSEG;
        t1 = min(p.seg_off[lo + 1], t0 + RSEG);
        s = p.seg_slot[lo];
      } else {
        t0 = p.segs[1 + sg];
        t1 = sg + 1 < nseg ? p.segs[2 + sg] : p.M;
        s = p.sslot[t0];
      }
      const int nrows = t1 - t0;  // 1..RSEG rows sharing one slot
      int32_t rank = 0, bad = 0;
      float scale = 0.f;
      if (s >= 0 && s < pl.num_slots) {
        rank = pl.rank[s];
        scale = pl.scale[s];
        if (rank < 1 || rank > pl.r_max) bad = MLORA_STATUS_BAD_RANK;
      } else if (s != -1) {
        bad = MLORA_STATUS_BAD_SLOT;
      }
      const int32_t *a_tr = nullptr, *b_tr = nullptr;
      if (pl.kind == MLORA_POOL_PAGED && s >= 0 && !bad) {
        // the slot's page ids, checked and kept in shared memory: every copy's address reads them there
        const int64_t tb = ((int64_t)s * pl.num_layers + pr.layer) * pl.r_max;
        const int32_t *ga = pl.a_tab + tb * pl.a_ppv, *gb = pl.b_tab + tb * pl.b_ppv;
        int32_t *pt = reinterpret_cast<int32_t *>(smem + S.pt) + q * p.ptn;
        const int na = rank * pl.a_ppv, nb = rank * pl.b_ppv;
        int32_t badp = 0;
        for (int e = lane; e < na + nb; e += 32) {
          const int32_t pg = e < na ? ga[e] : gb[e - na];
          badp |= (pg < 0) | (pg >= pl.num_pages);
          pt[e] = pg;
        }
        if (__any_sync(0xffffffffu, badp)) bad = MLORA_STATUS_BAD_PAGE;
        a_tr = pt;
        b_tr = pt + na;
      }
      const bool valid = s >= 0 && !bad;
      int32_t row = 0;
      if (lane < nrows) row = p.seg_off != nullptr ? t0 + lane : p.perm[t0 + lane];
      if (lane < RSEG) desc[q].rows[lane] = row;
      if (lane == 0) {
        desc[q].nrows = nrows;
        desc[q].rank = valid ? rank : 0;
        desc[q].bad = bad;
        desc[q].scale = scale;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&segfull[q]);
      if (!valid) continue;
      // the x slices of the segment's rows, once the consumers are done with the previous ones
      ok = __all_sync(0xffffffffu, (xuse == 0 || mbar_wait(xempty, (xuse - 1) & 1u, wlim)) && !*stop);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(xfull, (uint32_t)(nrows * (k1 - k0) * 2));
      __syncwarp();
      if (lane < nrows && k1 > k0)
        bulk_g2s(xbuf + lane * p.kpad, pr.x + (int64_t)row * pr.ldx + k0, (uint32_t)(k1 - k0) * 2, xfull);
      ++xuse;
      // the y rows' slices into L2, for the consumers' loads at the start of each chunk
      if (lane < nrows && n1 > n0) prefetch_l2(pr.y + (int64_t)row * pr.ldy + n0, (uint32_t)(n1 - n0) * 2);
      const int groups = (rank + ROWS - 1) / ROWS, bgroups = (rank + BROWS - 1) / BROWS;
      // this segment's stages: A^T (groups of 8 rank-rows, then d_in chunks of 4096), then B (d_out
      // chunks of 2048, then groups of 16 rank-rows)
      for (int ph = 0; ph < 2 && ok; ++ph) {
        const int outer = ph == 0 ? groups : nchunks, inner = ph == 0 ? kchunks : bgroups;
        const int srows = ph == 0 ? ROWS : BROWS, schunk = ph == 0 ? ACHUNK : CHUNK;
        for (int o = 0; o < outer && ok; ++o) {
          for (int in = 0; in < inner; ++in) {
            const int g = ph == 0 ? o : in, ch = ph == 0 ? in : o;
            const int slot = (int)(ctr % NS);
            const uint32_t su = ctr / NS;
            ok = __all_sync(0xffffffffu, (su == 0 || mbar_wait(&empty[slot], (su - 1) & 1u, wlim)) && !*stop);
            if (!ok) break;
            const int e0 = (ph == 0 ? k0 : n0) + ch * schunk;
            const int len = min(schunk, (ph == 0 ? k1 : n1) - e0), nr8 = min(srows, rank - g * srows);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(nr8 * len * 2));
            __syncwarp();
            if (lane < nr8) {
              uint16_t *dst = reinterpret_cast<uint16_t *>(ring + (size_t)slot * STAGE_BYTES) + lane * schunk;
              const int j = g * srows + lane;
              if (ph == 0)
                decode::vec_pieces<true>(pl, s, pr.layer, j, e0, e0 + len, a_tr, [&](const uint16_t *src, int off, int n) {
                  bulk_g2s_hint(dst + off, src, (uint32_t)n * 2, &full[slot], pol);
                });
              else
                decode::vec_pieces<false>(pl, s, pr.layer, j, e0, e0 + len, b_tr, [&](const uint16_t *src, int off, int n) {
                  bulk_g2s_hint(dst + off, src, (uint32_t)n * 2, &full[slot], pol);
                });
            }
            ++ctr;
          }
        }
      }
      if (!ok) break;
    }
    // Every copy issued lands before the CTA exits (after a normal run the consumers have waited
    // for all of them; after a time-out some may still be in flight).
    if (lane == 0) {
      if (!ok) {
        *stop = 1;
        report(p.status, MLORA_STATUS_TIMEOUT);
      }
      for (int i = 0; i < NS && (uint32_t)i < ctr; ++i) {
        const uint32_t cc = ctr - 1 - (uint32_t)i;  // the last stage issued into each slot
        (void)mbar_wait(&full[cc % NS], (cc / NS) & 1u, kDrainLimitNs);
      }
      if (xuse > 0) (void)mbar_wait(xfull, (xuse - 1) & 1u, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumer warps
    uint32_t ctr = 0;               // stages consumed
    uint32_t xuse = 0;              // valid segments consumed
    uint32_t vuse0 = 0, vuse1 = 0;  // valid segments that used exchange buffer 0 / 1
    bool ok = true;
    for (int i = 0;; ++i) {
      const int sg = snake(i, cb, C);
      if (sg >= nseg) break;
      const int q = i % RQ;
      const uint32_t use = (uint32_t)(i / RQ);
      ok = !consumers_or(!(!*stop && mbar_wait(&segfull[q], use & 1u, wlim)));
      if (!ok) break;
      const int nrows = desc[q].nrows, rank = desc[q].rank;
      const float scale = desc[q].scale;
      if (rank == 0) {
        if (c == 0 && tid == 0 && desc[q].bad) report(p.status, desc[q].bad);
        __syncwarp();
        if (lane == 0) mbar_arrive(&segempty[q]);
        continue;
      }
      const uint32_t vu = q == 0 ? vuse0++ : vuse1++;  // the use of exchange buffer q by valid segments
      // the segment's work with its row count rounded up to a power of two (the accumulators and
      // unrolled row loops sized at compile time; rows past nrows are skipped)
      auto segment = [&](auto rows_c) {
        constexpr int R = decltype(rows_c)::value;
        const int groups = (rank + ROWS - 1) / ROWS;
        // shrink over this CTA's slice of d_in: partial v[r][j], warp w owning rank-row 8 g + w
        if (cs > 1 && vu > 0) ok = __all_sync(0xffffffffu, mbar_wait(&vempty[q], (vu - 1) & 1u, wlim));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(xfull, xuse & 1u, wlim));
        ++xuse;
        if (cs > 1 && tid == 0) mbar_arrive_expect_tx(&vfull[q], (uint32_t)((cs - 1) * nrows * rank * 4));
        float *vmine = vx + (q * MAX_CS + c) * RSEG * MAX_RANK;  // [RSEG][MAX_RANK]
        // Warp w owns the 16-byte pieces 256 u + 32 w + lane (u = 0, 1) of every 4096-element chunk:
        // it loads each row's x pieces once per stage into registers and dots them with the pieces
        // of each of the stage's rank-rows
        // (one fp32 chain per rank-row and row). After the group's last chunk the chains are summed
        // over the lanes (scattered: lane l keeps value l / (32 / N)) into the group's slot in shared
        // memory; once every group is in, the warps' sums are added in warp order. No barrier
        // couples the warps inside the loop.
        constexpr int N = ROWS * R;  // values per lane: index jj * R + r
        for (int g = 0; g < groups && ok; ++g) {
          const int nr8 = min(ROWS, rank - g * ROWS);
          float acc[N];
  #pragma unroll
          for (int k = 0; k < N; ++k) acc[k] = 0.f;
          for (int ch = 0; ch < kchunks && ok; ++ch) {
            const int slot = (int)(ctr % NS);
            if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (ctr / NS) & 1u, wlim) && !*stop)) {
              ok = false;
              break;
            }
            const int e0 = ch * ACHUNK, len8 = min(ACHUNK, k1 - k0 - e0) >> 3;
  #pragma unroll
            for (int u = 0; u < ACHUNK / 2048; ++u) {
              const int c8 = u * 256 + warp * 32 + lane;  // 16-byte pieces, consecutive across the lanes
              if (c8 < len8) {
                uint4 xr[R];
  #pragma unroll
                for (int r = 0; r < R; ++r)
                  xr[r] = r < nrows ? *reinterpret_cast<const uint4 *>(xbuf + r * p.kpad + e0 + c8 * 8) : make_uint4(0u, 0u, 0u, 0u);
                const uint16_t *ar = reinterpret_cast<const uint16_t *>(ring + (size_t)slot * STAGE_BYTES) + c8 * 8;
  #pragma unroll
                for (int jj = 0; jj < ROWS; ++jj) {
                  if (jj < nr8) {
                    const uint4 av = *reinterpret_cast<const uint4 *>(ar + jj * ACHUNK);
  #pragma unroll
                    for (int r = 0; r < R; ++r)
                      if (r < nrows) mfma8_chain<DT>(xr[r], av, acc[jj * R + r]);
                  }
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            ++ctr;
          }
          if (ok) {
            const float tot = lane_sum_scatter<N>(acc, lane);
            float *red = reinterpret_cast<float *>(smem + S.red) + g * CWARPS * 32;
            if ((lane & (32 / N - 1)) == 0) red[warp * 32 + lane / (32 / N)] = tot;
          }
        }
        ok = !consumers_or(!ok);  // every group's sums are in (or some warp gave up)
        if (ok) {
          const float *red = reinterpret_cast<const float *>(smem + S.red);
          for (int e = tid; e < groups * N; e += CWARPS * 32) {
            const int g = e / N, k = e % N, jj = k / R, r = k % R, j = g * ROWS + jj;
            if (j < rank && r < nrows) {
              float v = 0.f;
              for (int w = 0; w < CWARPS; ++w) v += red[(g * CWARPS + w) * 32 + k];
              // this CTA's partial into slot c of every CTA's exchange buffer
              vmine[r * MAX_RANK + j] = v;
              for (int pe = 1; pe < cs; ++pe) {
                const uint32_t peer = (uint32_t)((c + pe) % cs);
                st_async_f32(dsmem_addr(vmine + r * MAX_RANK + j, peer), v, dsmem_addr(&vfull[q], peer));
              }
            }
          }
        }
        // the x slices may be refilled once every consumer is past the shrink
        ok = !consumers_or(!ok);
        if (lane == 0) mbar_arrive(xempty);
        if (ok && cs > 1) ok = !consumers_or(!mbar_wait_cluster(&vfull[q], vu & 1u, wlim));
        if (ok) {
          for (int e = tid; e < nrows * MAX_RANK; e += CWARPS * 32) {  // the cluster's partials, in CTA-rank order
            const int r = e / MAX_RANK, j = e % MAX_RANK;
            if (j < rank) {
              float v = 0.f;
              for (int cc = 0; cc < cs; ++cc) v += vx[((q * MAX_CS + cc) * RSEG + r) * MAX_RANK + j];
              vsm[r * MAX_RANK + j] = v;
            }
          }
        }
        ok = !consumers_or(!ok);  // v complete for every consumer, and this CTA's exchange buffer read
        if (ok && cs > 1 && tid == 0)
          for (int pe = 1; pe < cs; ++pe) mbar_arrive_remote(dsmem_addr(&vempty[q], (uint32_t)((c + pe) % cs)));
        // expand over this CTA's slice of d_out: y[n] = rn(y[n] + scale * sum_j v[j] B[j][n]), thread t
        // owning columns 8t.. of a chunk for every row of the segment
        for (int ch = 0; ch < nchunks && ok; ++ch) {
          const int nl = ch * CHUNK + tid * 8;  // column within the slice
          const bool mine = n0 + nl < n1;
          uint4 yw[R];  // this thread's y values, loaded before the chunk's stages are waited for
  #pragma unroll
          for (int r = 0; r < R; ++r)
            yw[r] = (mine && r < nrows) ? ldg_u4(pr.y + (int64_t)desc[q].rows[r] * pr.ldy + n0 + nl) : make_uint4(0u, 0u, 0u, 0u);
          float2 acc[R][4];
  #pragma unroll
          for (int r = 0; r < R; ++r)
  #pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][e] = make_float2(0.f, 0.f);
          const int bgroups = (rank + BROWS - 1) / BROWS;
          for (int g = 0; g < bgroups; ++g) {
            const int slot = (int)(ctr % NS);
            if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (ctr / NS) & 1u, wlim) && !*stop)) {
              ok = false;
              break;
            }
            const int nr8 = min(BROWS, rank - g * BROWS);
            if (mine) {
              const uint16_t *br = reinterpret_cast<const uint16_t *>(ring + (size_t)slot * STAGE_BYTES) + tid * 8;
              for (int w = 0; w < nr8; ++w) {
                float2 b2[4];
                unpack8x2<DT>(*reinterpret_cast<const uint4 *>(br + w * CHUNK), b2);
  #pragma unroll
                for (int r = 0; r < R; ++r) {
                  if (r < nrows) {
                    const float vj = vsm[r * MAX_RANK + g * BROWS + w];
                    const float2 v2 = make_float2(vj, vj);
  #pragma unroll
                    for (int e = 0; e < 4; ++e) acc[r][e] = __ffma2_rn(v2, b2[e], acc[r][e]);
                  }
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            ++ctr;
          }
          if (ok && mine) {
  #pragma unroll
            for (int r = 0; r < R; ++r) {
              if (r < nrows) {
                float yf[8];
                unpack8<DT>(yw[r], yf);
  #pragma unroll
                for (int e = 0; e < 4; ++e) {
                  yf[2 * e] = fmaf(scale, acc[r][e].x, yf[2 * e]);
                  yf[2 * e + 1] = fmaf(scale, acc[r][e].y, yf[2 * e + 1]);
                }
                *reinterpret_cast<uint4 *>(pr.y + (int64_t)desc[q].rows[r] * pr.ldy + n0 + nl) = pack8<DT>(yf);
              }
            }
          }
        }
      };
      if (nrows <= 1) segment(std::integral_constant<int, 1>{});
      else if (nrows <= 2 || RSEG == 2) segment(std::integral_constant<int, 2>{});
      else segment(std::integral_constant<int, RSEG>{});
      // every consumer is done with v and the descriptor before the producer may refill them
      ok = !consumers_or(!ok);
      if (!ok) break;
      if (lane == 0) mbar_arrive(&segempty[q]);
    }
    if (!ok && tid == 0) {
      *stop = 1;
      report(p.status, MLORA_STATUS_TIMEOUT);
      // partial sums the peers may still push land before the cluster leaves
      if (cs > 1)
        for (int b = 0; b < RQ; ++b) {
          const uint32_t n = b == 0 ? vuse0 : vuse1;
          if (n > 0) (void)mbar_wait_cluster(&vfull[b], (n - 1) & 1u, kDrainLimitNs);
        }
    }
  }
  __syncwarp();
  if (cs > 1) cluster_sync();  // no CTA leaves while a peer may still push into it or arrive on it
}

}  // namespace bstream

// CTAs per segment: two when a full-rank row's A^T and B exceed 1 MB (a lone SM streams about
// 50-100 GB/s), else one.
int stream_ctas(const PoolDev &pool) {
  const int64_t row = (int64_t)pool.r_max * (pool.d_in + pool.d_out) * 2;
  return row > 1024 * 1024 ? bstream::MAX_CS : 1;
}

bool stream_eligible(const PoolDev &pool, int num_rows) {
  if (pool.r_max < 32 || pool.r_max > bstream::MAX_RANK || num_rows < 1 || num_rows > kPlanMaxRows) return false;
  const int cs = stream_ctas(pool);
  const int kc = ((pool.d_in + cs - 1) / cs + 7) & ~7;
  const int kpad = (kc + bstream::CHUNK - 1) / bstream::CHUNK * bstream::CHUNK;
  const int ptn = pool.kind == MLORA_POOL_PAGED ? pool.r_max * (pool.a_ppv + pool.b_ppv) : 0;
  return ptn <= bstream::MAX_PT &&
         bstream::Smem::make(kpad, ptn, 2, (pool.r_max + bstream::ROWS - 1) / bstream::ROWS).total <= 227 * 1024;
}

static cudaError_t launch_stream(StreamParams p, cudaStream_t stream) {
  using namespace bstream;
  const ProblemDev &pr = p.pr;
  const int32_t M = p.M;
  p.cs = stream_ctas(pr.pool);
  p.kc = ((pr.pool.d_in + p.cs - 1) / p.cs + 7) & ~7;
  p.nc = ((pr.pool.d_out + p.cs - 1) / p.cs + 7) & ~7;
  p.kpad = (p.kc + CHUNK - 1) / CHUNK * CHUNK;
  p.ptn = pr.pool.kind == MLORA_POOL_PAGED ? pr.pool.r_max * (pr.pool.a_ppv + pr.pool.b_ppv) : 0;
  if (p.ptn > MAX_PT || pr.pool.r_max > MAX_RANK || (p.seg_off != nullptr && p.nseg > kStreamMaxSegs))
    return cudaErrorInvalidValue;
  const int gmax = (pr.pool.r_max + ROWS - 1) / ROWS;
  const int fixed = Smem::make(p.kpad, p.ptn, 0, gmax).total;
  int stages = (227 * 1024 - fixed) / STAGE_BYTES;
  stages = stages > MAX_STAGES ? MAX_STAGES : stages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  const size_t smem = (size_t)Smem::make(p.kpad, p.ptn, stages, gmax).total;
  auto kern = pr.pool.dtype == MLORA_BF16 ? stream_kernel<MLORA_BF16> : stream_kernel<MLORA_FP16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one CTA per SM; as many clusters of cs as can be resident at once (a GPC's SMs past a multiple
  // of cs stay idle), no more than there are rows
  const int sms = sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms / p.cs * p.cs), 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = sms / p.cs;
  if (p.cs > 1) {
    int resident = 0;
    if (cudaOccupancyMaxActiveClusters(&resident, (const void *)kern, &cfg) == cudaSuccess && resident > 0)
      clusters = resident < clusters ? resident : clusters;
  }
  clusters = clusters < M ? clusters : M;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3((unsigned)(clusters * p.cs), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_bgmv_stream(const ProblemDev &pr, const int32_t *perm, const int32_t *sslot, const int32_t *segs,
                               int32_t M, int32_t *status, uint64_t wait_ns, cudaStream_t stream) {
  StreamParams p{};
  p.pr = pr;
  p.perm = perm;
  p.sslot = sslot;
  p.segs = segs;
  p.M = M;
  p.status = status;
  p.wait_ns = wait_ns;
  return launch_stream(p, stream);
}

cudaError_t launch_sgmv_stream(const ProblemDev &pr, const int32_t *seg_off, const int32_t *seg_slot, int32_t nseg,
                               int32_t tc_min, int32_t M, int32_t *status, uint64_t wait_ns, cudaStream_t stream) {
  StreamParams p{};
  p.pr = pr;
  p.seg_off = seg_off;
  p.seg_slot = seg_slot;
  p.nseg = nseg;
  p.tc_min = tc_min;
  p.M = M;
  p.status = status;
  p.wait_ns = wait_ns;
  return launch_stream(p, stream);
}

}  // namespace mlora
