// bgmv_stream.cu -- BGMV rows of a heterogeneous-rank pool streamed through shared-memory rings
// (sm_103a, CUDA cores).
//
// S-LoRA serves thousands of adapters of different ranks from one paged pool and batches their
// decode rows together (S-LoRA section 3, "Heterogeneous Batching Kernels" and "Unified
// Paging"): a rank-64 row moves eight times the bytes of a rank-8 row. After the device-side
// grouping (bgmv_plan.cu: rows by rank, largest first, then by slot) this kernel gives each row to
// a cluster of cs CTAs. CTA c of the cluster streams its slice c of d_in of the row's A^T
// rank-rows, then its slice c of d_out of the B rank-rows, through a ring of shared-memory
// stages filled by bulk copies, so every CTA keeps up to 160 KB in flight whatever the row's rank
// and never reloads operands from L2 after a wait:
//   * one producer warp per CTA resolves each row (slot, rank, scale, page ids, checked),
//     publishes it in a row descriptor and issues the bulk copies: the slices of the x and y rows
//     into double buffers, then the stages -- a stage is 8 rank-rows x 2048 elements (32 KB): A^T's
//     row groups for every chunk of the d_in slice, then B's row groups for every chunk of the
//     d_out slice;
//   * eight consumer warps: for an A stage, warp w dots rank-row 8g + w's chunk with x's (mixed-
//     precision FMAs, fp32 sums, two chains per lane) and sums its lanes after the group's last
//     chunk (Punica section 3.4, the shrink, split over d_in); the cluster's partial sums are
//     pushed into every peer's shared memory (st.async, completing on the receiver's mbarrier) and
//     summed in CTA-rank order; for a B stage, thread t accumulates its 8 columns over the group's
//     rank-rows (paired fp32 FMAs) and, after the chunk's last group, writes y = rn(y + scale * sum)
//     (the expand, split over d_out);
//   * the stages cycle through full / empty mbarriers. Every wait is bounded: a CTA that gives up
//     reports MLORA_STATUS_TIMEOUT, stops issuing and, before it exits, waits (bounded) for the
//     copies it issued and the partial sums its peers may still push.
// The persistent grid of clusters takes the grouped rows in snake order (cluster b gets rows b,
// 2C - 1 - b, 2C + b, ... of C clusters), which balances the rows' sizes, largest first. Rows
// without adapter are skipped (y untouched); invalid slots, ranks and page ids are reported and
// their rows skipped. The sums run in a fixed order (a call is deterministic); it is another order
// than the decode kernel's, within the same tolerance.
#include <cuda_runtime.h>

#include "decode_impl.cuh"
#include "launch.h"

namespace mlora {
namespace bstream {

constexpr int CWARPS = 8;                    // consumer warps
constexpr int NTHREADS = (CWARPS + 1) * 32;  // + the producer warp
constexpr int ROWS = 8;                      // rank-rows per stage
constexpr int CHUNK = 2048;                  // elements of each rank-row per stage
constexpr int STAGE_BYTES = ROWS * CHUNK * 2;
constexpr int RQ = 2;                        // rows in flight (descriptors, x, y and exchange buffers)
constexpr int MAX_STAGES = 8;
constexpr int MAX_RANK = 128;
constexpr int MAX_CS = 4;                    // CTAs per row (cluster)
constexpr int MAX_PT = 2048;                 // page-table entries of one row kept in shared memory

struct RowDesc {
  int32_t row, rank, bad, slot;
  float scale;
  int32_t pad;
};

// Shared memory: [0, 512) barriers, [512, 1024) RQ row descriptors and the stop flag,
// [1024, 5120) vx [RQ][MAX_CS][MAX_RANK] fp32 partial v of every CTA of the cluster,
// [5120, 5632) vsm [MAX_RANK] the summed v, then the page ids of the rows in flight [RQ][ptn]
// (paged pools: the producer reads a row's page-table entries once, when it checks them), the x
// slices [RQ][kpad], the y slices [RQ][npad], the ring.
struct Smem {
  int pt, x, y, ring, total;
  __host__ __device__ static Smem make(int kpad, int npad, int ptn, int stages) {
    Smem s;
    s.pt = 5632;
    s.x = (s.pt + RQ * ptn * 4 + 127) & ~127;
    s.y = (s.x + RQ * kpad * 2 + 127) & ~127;
    s.ring = (s.y + RQ * npad * 2 + 1023) & ~1023;
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

// Row i of cluster b of C in snake order.
__device__ __forceinline__ int snake_row(int i, int b, int C) { return i * C + ((i & 1) ? C - 1 - b : b); }

template <int DT>
__global__ void __launch_bounds__(NTHREADS, 1) stream_kernel(const __grid_constant__ StreamParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [MAX_STAGES]
  uint64_t *empty = full + MAX_STAGES;                   // [MAX_STAGES]
  uint64_t *rowfull = empty + MAX_STAGES;                // [RQ]
  uint64_t *rowempty = rowfull + RQ;                     // [RQ]
  uint64_t *xfull = rowempty + RQ;                       // [RQ]
  uint64_t *yfull = xfull + RQ;                          // [RQ]
  uint64_t *vfull = yfull + RQ;                          // [RQ] the peers' partial sums landed
  uint64_t *vempty = vfull + RQ;                         // [RQ] the peers consumed this CTA's partial sums
  RowDesc *desc = reinterpret_cast<RowDesc *>(smem + 512);
  volatile int32_t *stop = reinterpret_cast<volatile int32_t *>(smem + 512 + RQ * sizeof(RowDesc));
  float *vx = reinterpret_cast<float *>(smem + 1024);
  float *vsm = reinterpret_cast<float *>(smem + 5120);
  const Smem S = Smem::make(p.kpad, p.npad, p.ptn, p.stages);
  uint16_t *xbuf = reinterpret_cast<uint16_t *>(smem + S.x);
  uint16_t *ybuf = reinterpret_cast<uint16_t *>(smem + S.y);
  uint8_t *ring = smem + S.ring;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const ProblemDev &pr = p.pr;
  const PoolDev &pl = pr.pool;
  const int cs = p.cs, NS = p.stages;
  const int c = cs > 1 ? (int)cluster_ctarank() : 0;
  const int cb = (int)blockIdx.x / cs, C = (int)gridDim.x / cs;  // this cluster, the clusters
  // this CTA's slices of d_in and d_out
  const int k0 = min(c * p.kc, pl.d_in), k1 = min(k0 + p.kc, pl.d_in);
  const int n0 = min(c * p.nc, pl.d_out), n1 = min(n0 + p.nc, pl.d_out);
  const int kchunks = (k1 - k0 + CHUNK - 1) / CHUNK, nchunks = (n1 - n0 + CHUNK - 1) / CHUNK;
  const uint64_t wlim = p.wait_ns ? p.wait_ns : kWaitLimitNs;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CWARPS);
    }
    for (int q = 0; q < RQ; ++q) {
      mbar_init(&rowfull[q], 1);
      mbar_init(&rowempty[q], CWARPS);
      mbar_init(&xfull[q], 1);
      mbar_init(&yfull[q], 1);
      mbar_init(&vfull[q], 1);
      mbar_init(&vempty[q], cs > 1 ? cs - 1 : 1);
    }
    *stop = 0;
    mbar_fence_init();
  }
  // x past the slice is zero in both buffers (the copies write [0, k1 - k0) only): a chunk's tail
  // then adds nothing, whatever stale bytes its stage holds (those are masked on the A side too)
  for (int e = (k1 - k0) + tid * 8; e < p.kpad; e += NTHREADS * 8)
    for (int q = 0; q < RQ; ++q) *reinterpret_cast<uint4 *>(xbuf + q * p.kpad + e) = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (cs > 1) cluster_sync();  // every peer's barriers are initialised before anything is pushed

  if (warp == CWARPS) {
    // ------------------------------------------------------------------ producer warp
    const uint64_t pol = policy_evict_first();
    uint32_t ctr = 0;                   // stages issued
    uint32_t xy_issued[RQ] = {0u, 0u};  // x / y copies issued into each buffer
    bool ok = true;
    for (int i = 0;; ++i) {
      const int t = snake_row(i, cb, C);
      if (t >= p.M) break;
      const int q = i % RQ;
      const uint32_t use = (uint32_t)(i / RQ);
      ok = __all_sync(0xffffffffu, (use == 0 || mbar_wait(&rowempty[q], (use - 1) & 1u, wlim)) && !*stop);
      if (!ok) break;
      int32_t row = 0, s = -1;
      if (lane == 0) {
        row = p.perm[t];
        s = p.sslot[t];
      }
      row = __shfl_sync(0xffffffffu, row, 0);
      s = __shfl_sync(0xffffffffu, s, 0);
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
        // the row's page ids, checked and kept in shared memory: every copy's address reads them there
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
      if (lane == 0) {
        desc[q].row = row;
        desc[q].rank = valid ? rank : 0;
        desc[q].bad = bad;
        desc[q].slot = s;
        desc[q].scale = scale;
        mbar_arrive(&rowfull[q]);
      }
      if (!valid) continue;
      if (lane == 0) {
        mbar_arrive_expect_tx(&xfull[q], (uint32_t)(k1 - k0) * 2);
        if (k1 > k0) bulk_g2s(xbuf + q * p.kpad, pr.x + (int64_t)row * pr.ldx + k0, (uint32_t)(k1 - k0) * 2, &xfull[q]);
        mbar_arrive_expect_tx(&yfull[q], (uint32_t)(n1 - n0) * 2);
        if (n1 > n0) bulk_g2s(ybuf + q * p.npad, pr.y + (int64_t)row * pr.ldy + n0, (uint32_t)(n1 - n0) * 2, &yfull[q]);
      }
      ++xy_issued[q];
      const int groups = (rank + ROWS - 1) / ROWS;
      // this row's stages: A^T (group-major, then d_in chunks), then B (d_out chunks, then groups)
      for (int ph = 0; ph < 2 && ok; ++ph) {
        const int outer = ph == 0 ? groups : nchunks, inner = ph == 0 ? kchunks : groups;
        for (int o = 0; o < outer && ok; ++o) {
          for (int in = 0; in < inner; ++in) {
            const int g = ph == 0 ? o : in, ch = ph == 0 ? in : o;
            const int slot = (int)(ctr % NS);
            const uint32_t su = ctr / NS;
            ok = __all_sync(0xffffffffu, (su == 0 || mbar_wait(&empty[slot], (su - 1) & 1u, wlim)) && !*stop);
            if (!ok) break;
            const int e0 = (ph == 0 ? k0 : n0) + ch * CHUNK;
            const int len = min(CHUNK, (ph == 0 ? k1 : n1) - e0), nrows = min(ROWS, rank - g * ROWS);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(nrows * len * 2));
            __syncwarp();
            if (lane < nrows) {
              uint16_t *dst = reinterpret_cast<uint16_t *>(ring + (size_t)slot * STAGE_BYTES) + lane * CHUNK;
              const int j = g * ROWS + lane;
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
      for (int b = 0; b < RQ; ++b) {
        if (xy_issued[b] == 0) continue;
        (void)mbar_wait(&xfull[b], (xy_issued[b] - 1) & 1u, kDrainLimitNs);
        (void)mbar_wait(&yfull[b], (xy_issued[b] - 1) & 1u, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumer warps
    uint32_t ctr = 0;               // stages consumed
    uint32_t used0 = 0, used1 = 0;  // valid rows that used buffer set 0 / 1
    bool ok = true;
    for (int i = 0;; ++i) {
      const int t = snake_row(i, cb, C);
      if (t >= p.M) break;
      const int q = i % RQ;
      const uint32_t use = (uint32_t)(i / RQ);
      ok = !consumers_or(!(!*stop && mbar_wait(&rowfull[q], use & 1u, wlim)));
      if (!ok) break;
      const RowDesc d = desc[q];
      if (d.rank == 0) {
        if (c == 0 && tid == 0 && d.bad) report(p.status, d.bad);
        __syncwarp();
        if (lane == 0) mbar_arrive(&rowempty[q]);
        continue;
      }
      const uint32_t vu = q == 0 ? used0++ : used1++;  // the use of buffer set q by valid rows
      const int groups = (d.rank + ROWS - 1) / ROWS;
      // shrink over this CTA's slice of d_in: v[j] partial, warp w owning rank-row 8 g + w
      if (cs > 1 && vu > 0) ok = __all_sync(0xffffffffu, mbar_wait(&vempty[q], (vu - 1) & 1u, wlim));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&xfull[q], vu & 1u, wlim));
      if (cs > 1 && tid == 0) mbar_arrive_expect_tx(&vfull[q], (uint32_t)((cs - 1) * d.rank * 4));
      const uint16_t *xr = xbuf + q * p.kpad;
      float *vmine = vx + (q * MAX_CS + c) * MAX_RANK;
      for (int g = 0; g < groups && ok; ++g) {
        const int j = g * ROWS + warp;
        float c0 = 0.f, c1 = 0.f;
        for (int ch = 0; ch < kchunks; ++ch) {
          const int slot = (int)(ctr % NS);
          if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (ctr / NS) & 1u, wlim) && !*stop)) {
            ok = false;
            break;
          }
          if (j < d.rank) {
            const int e0 = ch * CHUNK, len8 = min(CHUNK, k1 - k0 - e0) >> 3;
            const uint16_t *ar = reinterpret_cast<const uint16_t *>(ring + (size_t)slot * STAGE_BYTES) + warp * CHUNK;
#pragma unroll
            for (int u = 0; u < CHUNK / 256; ++u) {
              const int c8 = u * 32 + lane;  // 16-byte pieces, consecutive across the lanes
              const uint4 av = c8 < len8 ? *reinterpret_cast<const uint4 *>(ar + c8 * 8) : make_uint4(0u, 0u, 0u, 0u);
              mfma8<DT>(*reinterpret_cast<const uint4 *>(xr + e0 + c8 * 8), av, c0, c1);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
          ++ctr;
        }
        if (ok && j < d.rank) {
          float v = c0 + c1;
#pragma unroll
          for (int sft = 16; sft > 0; sft >>= 1) v += __shfl_xor_sync(0xffffffffu, v, sft);
          // this CTA's partial into slot c of every CTA's exchange buffer
          if (lane == 0) {
            vmine[j] = v;
            for (int pe = 1; pe < cs; ++pe) {
              const uint32_t peer = (uint32_t)((c + pe) % cs);
              st_async_f32(dsmem_addr(vmine + j, peer), v, dsmem_addr(&vfull[q], peer));
            }
          }
        }
      }
      ok = !consumers_or(!ok);
      if (ok && cs > 1) ok = !consumers_or(!mbar_wait_cluster(&vfull[q], vu & 1u, wlim));
      if (ok) {
        for (int j = tid; j < d.rank; j += CWARPS * 32) {  // the cluster's partials, in CTA-rank order
          float v = 0.f;
          for (int cc = 0; cc < cs; ++cc) v += vx[(q * MAX_CS + cc) * MAX_RANK + j];
          vsm[j] = v;
        }
      }
      ok = !consumers_or(!ok);  // v complete for every consumer, and this CTA's exchange buffer read
      if (ok && cs > 1 && tid == 0)
        for (int pe = 1; pe < cs; ++pe) mbar_arrive_remote(dsmem_addr(&vempty[q], (uint32_t)((c + pe) % cs)));
      // expand over this CTA's slice of d_out: y[n] = rn(y[n] + scale * sum_j v[j] B[j][n]), thread t
      // owning columns 8t.. of a chunk
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&yfull[q], vu & 1u, wlim));
      const uint16_t *yr = ybuf + q * p.npad;
      for (int ch = 0; ch < nchunks && ok; ++ch) {
        float2 acc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.f, 0.f);
        const int nl = ch * CHUNK + tid * 8;  // column within the slice
        const bool mine = n0 + nl < n1;
        for (int g = 0; g < groups; ++g) {
          const int slot = (int)(ctr % NS);
          if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (ctr / NS) & 1u, wlim) && !*stop)) {
            ok = false;
            break;
          }
          const int nrows = min(ROWS, d.rank - g * ROWS);
          if (mine) {
            const uint16_t *br = reinterpret_cast<const uint16_t *>(ring + (size_t)slot * STAGE_BYTES) + tid * 8;
            for (int w = 0; w < nrows; ++w) {
              float2 b2[4];
              unpack8x2<DT>(*reinterpret_cast<const uint4 *>(br + w * CHUNK), b2);
              const float vj = vsm[g * ROWS + w];
              const float2 v2 = make_float2(vj, vj);
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[e] = __ffma2_rn(v2, b2[e], acc[e]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
          ++ctr;
        }
        if (ok && mine) {
          float yf[8];
          unpack8<DT>(*reinterpret_cast<const uint4 *>(yr + nl), yf);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            yf[2 * e] = fmaf(d.scale, acc[e].x, yf[2 * e]);
            yf[2 * e + 1] = fmaf(d.scale, acc[e].y, yf[2 * e + 1]);
          }
          *reinterpret_cast<uint4 *>(pr.y + (int64_t)d.row * pr.ldy + n0 + nl) = pack8<DT>(yf);
        }
      }
      // every consumer is done with v, x and y of this row before the producer may refill them
      ok = !consumers_or(!ok);
      if (!ok) break;
      if (lane == 0) mbar_arrive(&rowempty[q]);
    }
    if (!ok && tid == 0) {
      *stop = 1;
      report(p.status, MLORA_STATUS_TIMEOUT);
      // partial sums the peers may still push land before the cluster leaves
      if (cs > 1)
        for (int b = 0; b < RQ; ++b) {
          const uint32_t n = b == 0 ? used0 : used1;
          if (n > 0) (void)mbar_wait_cluster(&vfull[b], (n - 1) & 1u, kDrainLimitNs);
        }
    }
  }
  __syncwarp();
  if (cs > 1) cluster_sync();  // no CTA leaves while a peer may still push into it or arrive on it
}

}  // namespace bstream

// CTAs per row: the fewest (at most 4) that keep every CTA's share of a full-rank row's A^T and
// B slices within 1 MB (a lone SM streams about 50-100 GB/s).
int stream_ctas(const PoolDev &pool) {
  const int64_t row = (int64_t)pool.r_max * (pool.d_in + pool.d_out) * 2;
  int cs = 1;
  while (cs < bstream::MAX_CS && row / cs > 1024 * 1024) cs <<= 1;
  return cs;
}

// Batches of up to four rows per SM: with more, rows that share an adapter are the rule (Zipf
// popularity) and the decode kernel's grouped order reads each adapter's rows from L2 for less.
// (Llama-2-70B q_proj, 2000 adapters of ranks 8..64, Zipf 1.2: 256 rows 85.6 -> 61.2 us streamed,
// 2048 rows 354 us grouped on the decode kernel against 385 us streamed.)
bool stream_eligible(const PoolDev &pool, int num_rows) {
  if (pool.r_max < 32 || pool.r_max > bstream::MAX_RANK || num_rows < 1 || num_rows > 4 * sm_count()) return false;
  const int cs = stream_ctas(pool);
  const int kc = ((pool.d_in + cs - 1) / cs + 7) & ~7, nc = ((pool.d_out + cs - 1) / cs + 7) & ~7;
  const int kpad = (kc + bstream::CHUNK - 1) / bstream::CHUNK * bstream::CHUNK;
  const int ptn = pool.kind == MLORA_POOL_PAGED ? pool.r_max * (pool.a_ppv + pool.b_ppv) : 0;
  return ptn <= bstream::MAX_PT && bstream::Smem::make(kpad, nc, ptn, 2).total <= 227 * 1024;
}

cudaError_t launch_bgmv_stream(const ProblemDev &pr, const int32_t *perm, const int32_t *sslot, int32_t M,
                               int32_t *status, uint64_t wait_ns, cudaStream_t stream) {
  using namespace bstream;
  StreamParams p{};
  p.pr = pr;
  p.perm = perm;
  p.sslot = sslot;
  p.M = M;
  p.status = status;
  p.wait_ns = wait_ns;
  p.cs = stream_ctas(pr.pool);
  p.kc = ((pr.pool.d_in + p.cs - 1) / p.cs + 7) & ~7;
  p.nc = ((pr.pool.d_out + p.cs - 1) / p.cs + 7) & ~7;
  p.kpad = (p.kc + CHUNK - 1) / CHUNK * CHUNK;
  p.npad = p.nc;
  p.ptn = pr.pool.kind == MLORA_POOL_PAGED ? pr.pool.r_max * (pr.pool.a_ppv + pr.pool.b_ppv) : 0;
  if (p.ptn > MAX_PT || pr.pool.r_max > MAX_RANK) return cudaErrorInvalidValue;
  const int fixed = Smem::make(p.kpad, p.npad, p.ptn, 0).total;
  int stages = (227 * 1024 - fixed) / STAGE_BYTES;
  stages = stages > MAX_STAGES ? MAX_STAGES : stages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  const size_t smem = (size_t)Smem::make(p.kpad, p.npad, p.ptn, stages).total;
  auto kern = pr.pool.dtype == MLORA_BF16 ? stream_kernel<MLORA_BF16> : stream_kernel<MLORA_FP16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (p.cs > 1) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
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

}  // namespace mlora
