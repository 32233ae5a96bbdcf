// decode_impl.cuh -- CUDA-core kernel for decode-sized row tiles (sm_103a); instantiated per
// mode by decode_shrink.cu, decode_expand.cu and decode_fused.cu.
//
// Work unit: a TILE = up to RT consecutive rows that use one adapter (a piece of an SGMV
// segment, or one BGMV row). The delta of a tile is a few dot products over d_in (shrink) and
// a few axpys over d_out (expand): matrix-vector work bound by memory, which runs on the CUDA
// cores (Punica section 3.4, "The degenerate case": one request per adapter is I/O-bound and
// uses coalesced CUDA-core loads rather than tensor cores).
//
// One CTA per (problem, tile, split). The grid is flat; CTAs of one tile form a cluster.
//   * Split-K shrink (Punica section 3.4, "SGMV-shrink schedule") across the cluster: each CTA
//     reduces its slice of d_in, then pushes its partial v into every peer's shared memory with
//     st.async; the pushes complete on the receiver's mbarrier, and every CTA sums the partials
//     in CTA-rank order. No grid-wide barrier, no workspace, no atomics, a fixed summation order.
//   * Output-split expand (Punica section 3.4, "SGMV-expand schedule"): each CTA owns a slice of
//     d_out, streams B[s] rows for that slice once per tile and rewrites y in place.
//   * FUSED mode does both in one launch; v never leaves the chip.
//   * Operands move by TMA bulk copies (cp.async.bulk) into a shared-memory ring of mbarrier
//     stages; warp 0 issues, all warps compute.
//   * Programmatic dependent launch (when the caller enables it): a kernel lets the next one in
//     the stream start at once.
//     Before griddepcontrol.wait a CTA only reads what no kernel of this library writes (the
//     rows' metadata, the pool, the page tables) and requests its adapter rows; x, y and v,
//     which the previous kernel may have written, are read after the wait. The adapter
//     weights -- most of the bytes -- therefore stream in while the previous kernel finishes.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace mlora {
namespace decode {

constexpr int NTHREADS = 256;
constexpr int NWARPS = NTHREADS / 32;
constexpr int MAX_STAGES = 4;
constexpr int SCAN_CAP = 1024;  // segment offsets staged per scan round
constexpr int MAX_CS = 16;      // CTAs per tile (cluster size)

struct TileInfo {
  int32_t row0, nr, slot, rank;
  float scale;
  int32_t skip;  // nonzero: nothing to do for this tile
  int32_t bad;   // status bits found while resolving
  int32_t pad;
};

__device__ __forceinline__ const uint16_t *a_row(const PoolDev &pl, int s, int layer, int j) {
  const int64_t t = ((int64_t)s * pl.num_layers + layer) * pl.r_max + j;
  if (pl.kind == MLORA_POOL_STACKED) return pl.a_t + t * pl.d_in;
  return pl.pages + (int64_t)pl.a_tab[t] * pl.page_elems;
}

__device__ __forceinline__ const uint16_t *b_row(const PoolDev &pl, int s, int layer, int j) {
  const int64_t t = ((int64_t)s * pl.num_layers + layer) * pl.r_max + j;
  if (pl.kind == MLORA_POOL_STACKED) return pl.b + t * pl.d_out;
  return pl.pages + (int64_t)pl.b_tab[t] * pl.page_elems;
}

// Resolve virtual tile `t` of problem `pr` into `ti` (whole block participates; reads only
// metadata that no kernel of this library writes).
// SGMV: segments contribute ceil(len / rt) tiles each, in segment order. BGMV: tile t is row t.
template <int MODE>
__device__ void resolve_tile(const DecodeParams &p, const ProblemDev &pr, int t, TileInfo *ti, int32_t *scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    ti->skip = 1;
    ti->bad = 0;
    ti->nr = 0;
  }
  __syncthreads();
  if (p.seg_off != nullptr) {
    int32_t carry = 0, found = 0, bad = 0;
    for (int base = 0; base < p.nseg; base += SCAN_CAP) {
      const int cnt = min(SCAN_CAP, p.nseg - base);
      for (int q = tid; q <= cnt; q += NTHREADS) scan[q] = p.seg_off[base + q];
      __syncthreads();
      if (warp == 0) {
        for (int q0 = 0; q0 < cnt; q0 += 32) {
          const int q = q0 + lane;
          int32_t len = 0, lo = 0;
          if (q < cnt) {
            lo = scan[q];
            len = scan[q + 1] - lo;
            if (len < 0 || lo < 0 || scan[q + 1] > p.M) bad = 1;
          }
          const int32_t nt = (q < cnt && len > 0) ? (len + p.rt - 1) / p.rt : 0;
          int32_t incl = nt;
#pragma unroll
          for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
          }
          const int32_t excl = carry + incl - nt;
          const bool mine = q < cnt && t >= excl && t < excl + nt;
          if (!found && mine) {
            const int32_t sub = t - excl;
            ti->row0 = lo + sub * p.rt;
            ti->nr = min(p.rt, len - sub * p.rt);
            ti->slot = p.seg_slot[base + q];
          }
          found |= __any_sync(0xffffffffu, mine);
          carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        bad = __any_sync(0xffffffffu, bad);
      }
      __syncthreads();
    }
    if (tid == 0) {
      const bool ends_ok = p.seg_off[0] == 0 && p.seg_off[p.nseg] == p.M;
      if (bad || !ends_ok) {
        ti->bad = MLORA_STATUS_BAD_OFFSETS;
        found = 0;
      }
      ti->skip = found ? 0 : 1;
    }
  } else if (tid == 0 && t < p.M) {
    ti->row0 = t;
    ti->nr = 1;
    ti->slot = p.row_slot[t];
    ti->skip = 0;
  }
  __syncthreads();
  // Adapter checks (warp 0): slot range, rank range, page ids of the rank-rows this mode reads.
  if (warp == 0 && !ti->skip) {
    const int s = ti->slot;
    const PoolDev &pl = pr.pool;
    int32_t bad = 0, skip = 0, rank = 0;
    float scale = 0.f;
    if (s == -1) {
      skip = 1;
    } else if (s < -1 || s >= pl.num_slots) {
      bad = MLORA_STATUS_BAD_SLOT;
    } else {
      rank = pl.rank[s];
      scale = pl.scale[s];
      if (rank < 1 || rank > pl.r_max) {
        bad = MLORA_STATUS_BAD_RANK;
      } else if (pl.kind == MLORA_POOL_PAGED) {
        const int64_t t0 = ((int64_t)s * pl.num_layers + pr.layer) * pl.r_max;
        int32_t badp = 0;
        for (int j = lane; j < rank; j += 32) {
          if (MODE != MODE_EXPAND) {
            const int32_t pg = pl.a_tab[t0 + j];
            badp |= (pg < 0 || pg >= pl.num_pages);
          }
          if (MODE != MODE_SHRINK) {
            const int32_t pg = pl.b_tab[t0 + j];
            badp |= (pg < 0 || pg >= pl.num_pages);
          }
        }
        if (__any_sync(0xffffffffu, badp)) bad = MLORA_STATUS_BAD_PAGE;
      }
    }
    if (lane == 0) {
      ti->rank = rank;
      ti->scale = scale;
      ti->bad |= bad;
      ti->skip = (skip || bad) ? 1 : 0;
    }
  }
  __syncthreads();
}

// Shared-memory layout (dynamic):
//   [0, 128)           mbarriers: full_k[4], full_e[4], xbar
//   [128, 160)         TileInfo
//   [256, ...)         gather buffer gbuf[cs][RT][r_alloc] floats (partial v of every CTA)
//                      vsm[RT][r_alloc] floats (summed v)
//                      scan[SCAN_CAP + 1] ints
//                      ring_k: sk stages of (r_alloc + RT) x kb elements (A rows, then x rows)
//                      ring_e: se stages of (r_alloc + RT) x nb elements (B rows, then y rows)
struct Layout {
  int gbuf, vsm, scan, ring_k, ring_e, total;
  __host__ __device__ static Layout make(int cs, int rt, int r_alloc, int sk, int kb, int se, int nb) {
    Layout L;
    L.gbuf = 256;
    L.vsm = L.gbuf + cs * rt * r_alloc * 4;
    L.scan = L.vsm + rt * r_alloc * 4;
    L.ring_k = (L.scan + (SCAN_CAP + 1) * 4 + 127) & ~127;
    L.ring_e = L.ring_k + sk * (r_alloc + rt) * kb * 2;
    L.total = L.ring_e + se * (r_alloc + rt) * nb * 2;
    return L;
  }
};

template <int DT, int MODE, int RT, int JPW>
__global__ void __launch_bounds__(NTHREADS) decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int cs = p.csplit;  // CTAs per tile: the cluster (SHRINK, FUSED) or the N-split (EXPAND)
  const Layout L = Layout::make(MODE == MODE_EXPAND ? 1 : cs, RT, p.r_alloc, p.sk, p.kb, p.se, p.nb);
  uint64_t *full_k = reinterpret_cast<uint64_t *>(smem);
  uint64_t *full_e = full_k + MAX_STAGES;
  uint64_t *xbar = full_e + MAX_STAGES;
  TileInfo *ti = reinterpret_cast<TileInfo *>(smem + 128);
  float *gbuf = reinterpret_cast<float *>(smem + L.gbuf);
  float *vsm = reinterpret_cast<float *>(smem + L.vsm);
  int32_t *scan = reinterpret_cast<int32_t *>(smem + L.scan);
  uint8_t *ring_k = smem + L.ring_k;
  uint8_t *ring_e = smem + L.ring_e;
  const int stage_k_elems = (p.r_alloc + RT) * p.kb;
  const int stage_e_elems = (p.r_alloc + RT) * p.nb;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool clustered = (MODE != MODE_EXPAND) && cs > 1;
  const uint32_t c = (MODE == MODE_EXPAND) ? (blockIdx.x % cs) : cluster_ctarank();
  const int64_t unit = blockIdx.x / cs;  // (problem, tile)
  const int prob = (int)(unit / p.tiles);
  const int t = (int)(unit % p.tiles);
  const ProblemDev &pr = p.prob[prob];
  const PoolDev &pl = pr.pool;

  if (tid == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&full_e[s], 1);
    }
    mbar_init(xbar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (clustered) cluster_arrive_relaxed();  // peers may push into our gbuf once everyone arrived
  pdl_launch_dependents();                  // the next kernel may start; it waits for us before reading our outputs

  resolve_tile<MODE>(p, pr, t, ti, scan);
  if (c == 0 && tid == 0 && ti->bad) report(p.status, ti->bad);
  const bool active = !ti->skip;  // uniform across the block and across the cluster
  const int row0 = ti->row0, nr = ti->nr, s = ti->slot, rank = ti->rank;
  const float scale = ti->scale;

  // This CTA's slices of d_in and d_out.
  const int kchunk = ((pl.d_in + cs - 1) / cs + 7) & ~7;
  const int nchunk = ((pl.d_out + cs - 1) / cs + 7) & ~7;
  const int k_begin = min((int)c * kchunk, pl.d_in), k_end = min(k_begin + kchunk, pl.d_in);
  const int n_begin = min((int)c * nchunk, pl.d_out), n_end = min(n_begin + nchunk, pl.d_out);
  const int nkb = (MODE == MODE_EXPAND || !active) ? 0 : (k_end - k_begin + p.kb - 1) / p.kb;
  const int nnb = (MODE == MODE_SHRINK || !active) ? 0 : (n_end - n_begin + p.nb - 1) / p.nb;
  const uint64_t evict_first = policy_evict_first();

  // Producer (warp 0). A stage's barrier expects its adapter rows and its activation rows; the
  // adapter rows may be requested before griddepcontrol.wait, the activation rows only after.
  auto expect_k = [&](int blk) {
    const int kv = min(p.kb, k_end - (k_begin + blk * p.kb));
    if (lane == 0) mbar_arrive_expect_tx(&full_k[blk % p.sk], (uint32_t)((rank + nr) * kv * 2));
  };
  auto issue_k = [&](int blk, bool weights, bool acts) {
    const int stage = blk % p.sk;
    const int k0 = k_begin + blk * p.kb, kv = min(p.kb, k_end - k0);
    uint16_t *base = reinterpret_cast<uint16_t *>(ring_k) + stage * stage_k_elems;
    for (int q = lane; q < rank + nr; q += 32) {
      if (q < rank) {
        if (weights) bulk_g2s_hint(base + q * p.kb, a_row(pl, s, pr.layer, q) + k0, kv * 2, &full_k[stage], evict_first);
      } else if (acts) {
        const int i = q - rank;
        bulk_g2s(base + (p.r_alloc + i) * p.kb, pr.x + (int64_t)(row0 + i) * pr.ldx + k0, kv * 2, &full_k[stage]);
      }
    }
  };
  auto expect_e = [&](int blk) {
    const int nv = min(p.nb, n_end - (n_begin + blk * p.nb));
    if (lane == 0) mbar_arrive_expect_tx(&full_e[blk % p.se], (uint32_t)((rank + nr) * nv * 2));
  };
  auto issue_e = [&](int blk, bool weights, bool acts) {
    const int stage = blk % p.se;
    const int n0 = n_begin + blk * p.nb, nv = min(p.nb, n_end - n0);
    uint16_t *base = reinterpret_cast<uint16_t *>(ring_e) + stage * stage_e_elems;
    for (int q = lane; q < rank + nr; q += 32) {
      if (q < rank) {
        if (weights) bulk_g2s_hint(base + q * p.nb, b_row(pl, s, pr.layer, q) + n0, nv * 2, &full_e[stage], evict_first);
      } else if (acts) {
        const int i = q - rank;
        bulk_g2s(base + (p.r_alloc + i) * p.nb, pr.y + (int64_t)(row0 + i) * pr.ldy + n0, nv * 2, &full_e[stage]);
      }
    }
  };

  const int pk = min(nkb, p.sk), pe = min(nnb, p.se);
  if (warp == 0) {
    if (clustered && lane == 0 && active) mbar_arrive_expect_tx(xbar, (uint32_t)(cs * nr * rank * 4));
    for (int b = 0; b < pk; ++b) {
      expect_k(b);
      __syncwarp();
      issue_k(b, true, false);
    }
    for (int b = 0; b < pe; ++b) {
      expect_e(b);
      __syncwarp();
      issue_e(b, true, false);
    }
  }
  pdl_wait();  // the previous kernel in the stream has finished; its writes are visible
  if (warp == 0) {
    for (int b = 0; b < pk; ++b) issue_k(b, false, true);
    for (int b = 0; b < pe; ++b) issue_e(b, false, true);
  }
  uint32_t issued_k = pk, issued_e = pe, done_k = 0, done_e = 0;
  int timed_out = 0;

  // ---------------- shrink: partial v over this CTA's slice of d_in ----------------
  if (MODE != MODE_EXPAND) {
    float acc[RT][JPW];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) acc[i][jj] = 0.f;

    for (int blk = 0; blk < nkb && !timed_out; ++blk) {
      const int stage = blk % p.sk;
      const int ok = mbar_wait(&full_k[stage], (uint32_t)(blk / p.sk) & 1u) ? 1 : 0;
      timed_out = __syncthreads_or(!ok);
      if (timed_out) break;
      ++done_k;
      const int kv = min(p.kb, k_end - (k_begin + blk * p.kb));
      const uint16_t *As = reinterpret_cast<const uint16_t *>(ring_k) + stage * stage_k_elems;
      const uint16_t *Xs = As + p.r_alloc * p.kb;
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) {
        const int j = warp + jj * NWARPS;
        if (j < rank) {
          const uint16_t *arow = As + j * p.kb;
          for (int c8 = lane; c8 < (kv >> 3); c8 += 32) {
            float af[8];
            unpack8<DT>(*reinterpret_cast<const uint4 *>(arow + c8 * 8), af);
#pragma unroll
            for (int i = 0; i < RT; ++i) {
              if (i < nr) {
                float xf[8];
                unpack8<DT>(*reinterpret_cast<const uint4 *>(Xs + i * p.kb + c8 * 8), xf);
                float sacc = acc[i][jj];
#pragma unroll
                for (int e = 0; e < 8; ++e) sacc = fmaf(xf[e], af[e], sacc);
                acc[i][jj] = sacc;
              }
            }
          }
        }
      }
      __syncthreads();  // stage consumed by every warp
      if (blk + p.sk < nkb) {
        if (warp == 0) {
          expect_k(blk + p.sk);
          __syncwarp();
          issue_k(blk + p.sk, true, true);
        }
        ++issued_k;
      }
    }

    // warp-level sum of each (row, rank) dot product: every lane ends with the total
#pragma unroll
    for (int jj = 0; jj < JPW; ++jj) {
#pragma unroll
      for (int i = 0; i < RT; ++i) {
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) acc[i][jj] += __shfl_xor_sync(0xffffffffu, acc[i][jj], d);
      }
    }

    if (clustered) {
      // Push this CTA's partials into slot c of every peer's gather buffer (lane q -> CTA q).
      cluster_wait();  // every peer has initialised its barriers
      if (active && !timed_out && lane < cs) {
        const uint32_t peer_gbuf = dsmem_addr(gbuf, lane);
        const uint32_t peer_bar = dsmem_addr(xbar, lane);
#pragma unroll
        for (int jj = 0; jj < JPW; ++jj) {
          const int j = warp + jj * NWARPS;
          if (j < rank) {
#pragma unroll
            for (int i = 0; i < RT; ++i) {
              if (i < nr) st_async_f32(peer_gbuf + 4u * (uint32_t)((c * RT + i) * p.r_alloc + j), acc[i][jj], peer_bar);
            }
          }
        }
      }
      if (active && !timed_out) {
        const int ok = mbar_wait_cluster(xbar, 0) ? 1 : 0;
        timed_out = __syncthreads_or(!ok);
      } else {
        __syncthreads();
      }
      if (active && !timed_out) {
        for (int e = tid; e < nr * rank; e += NTHREADS) {
          const int i = e / rank, j = e % rank;
          float sum = 0.f;
          for (int q = 0; q < cs; ++q) sum += gbuf[(q * RT + i) * p.r_alloc + j];
          if (MODE == MODE_SHRINK) {
            if (e % cs == (int)c) pr.v[(int64_t)(row0 + i) * pl.r_max + j] = sum;
          } else {
            vsm[i * p.r_alloc + j] = sum;
          }
        }
      }
    } else if (active && !timed_out && lane == 0) {
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) {
        const int j = warp + jj * NWARPS;
        if (j < rank) {
#pragma unroll
          for (int i = 0; i < RT; ++i) {
            if (i < nr) {
              if (MODE == MODE_SHRINK) pr.v[(int64_t)(row0 + i) * pl.r_max + j] = acc[i][jj];
              else vsm[i * p.r_alloc + j] = acc[i][jj];
            }
          }
        }
      }
    }
    __syncthreads();
  } else if (active) {
    // expand only: this tile's v rows from global memory (written by the previous kernel)
    for (int e = tid; e < nr * rank; e += NTHREADS) {
      const int i = e / rank, j = e % rank;
      vsm[i * p.r_alloc + j] = pr.v[(int64_t)(row0 + i) * pl.r_max + j];
    }
    __syncthreads();
  }

  // ---------------- expand: y[rows][this CTA's slice of d_out] ----------------
  if (MODE != MODE_SHRINK) {
    for (int blk = 0; blk < nnb && !timed_out; ++blk) {
      const int stage = blk % p.se;
      const int ok = mbar_wait(&full_e[stage], (uint32_t)(blk / p.se) & 1u) ? 1 : 0;
      timed_out = __syncthreads_or(!ok);
      if (timed_out) break;
      ++done_e;
      const int n0 = n_begin + blk * p.nb, nv = min(p.nb, n_end - n0);
      const uint16_t *Bs = reinterpret_cast<const uint16_t *>(ring_e) + stage * stage_e_elems;
      const uint16_t *Ys = Bs + p.r_alloc * p.nb;
      for (int c8 = tid; c8 < (nv >> 3); c8 += NTHREADS) {
        float acc[RT][8];
#pragma unroll
        for (int i = 0; i < RT; ++i)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
        for (int j = 0; j < rank; ++j) {
          float bf[8];
          unpack8<DT>(*reinterpret_cast<const uint4 *>(Bs + j * p.nb + c8 * 8), bf);
#pragma unroll
          for (int i = 0; i < RT; ++i) {
            if (i < nr) {
              const float vij = vsm[i * p.r_alloc + j];
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(vij, bf[e], acc[i][e]);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < RT; ++i) {
          if (i < nr) {
            float yf[8];
            unpack8<DT>(*reinterpret_cast<const uint4 *>(Ys + i * p.nb + c8 * 8), yf);
#pragma unroll
            for (int e = 0; e < 8; ++e) yf[e] = fmaf(scale, acc[i][e], yf[e]);
            *reinterpret_cast<uint4 *>(pr.y + (int64_t)(row0 + i) * pr.ldy + n0 + c8 * 8) = pack8<DT>(yf);
          }
        }
      }
      __syncthreads();
      if (blk + p.se < nnb) {
        if (warp == 0) {
          expect_e(blk + p.se);
          __syncwarp();
          issue_e(blk + p.se, true, true);
        }
        ++issued_e;
      }
    }
  }

  if (timed_out) {
    // Wait (bounded) for this CTA's copies still in flight before its shared memory goes away.
    for (uint32_t g = done_k; g < issued_k; ++g) (void)mbar_wait(&full_k[g % p.sk], (g / p.sk) & 1u, 100000000ull);
    for (uint32_t g = done_e; g < issued_e; ++g) (void)mbar_wait(&full_e[g % p.se], (g / p.se) & 1u, 100000000ull);
    if (tid == 0) report(p.status, MLORA_STATUS_TIMEOUT);
  }
  if (clustered) cluster_sync();  // no CTA leaves while a peer may still write into its shared memory
}

// Host: launch one instantiation with the cluster and PDL attributes.
template <int DT, int MODE, int RT, int JPW>
cudaError_t launch_one(const DecodeParams &p, unsigned grid, size_t smem, int cluster, bool pdl, cudaStream_t stream) {
  auto kern = decode_kernel<DT, MODE, RT, JPW>;
  static int configured_smem[64] = {0};  // per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured_smem[dev] < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = (int)smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (MODE != MODE_EXPAND) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int DT, int MODE>
cudaError_t dispatch(const DecodeParams &p, unsigned grid, size_t smem, int cluster, bool pdl, cudaStream_t stream) {
  const int r = p.r_alloc;
  if (p.rt == 1) {
    if (r <= 16) return launch_one<DT, MODE, 1, 2>(p, grid, smem, cluster, pdl, stream);
    if (r <= 32) return launch_one<DT, MODE, 1, 4>(p, grid, smem, cluster, pdl, stream);
    if (r <= 64) return launch_one<DT, MODE, 1, 8>(p, grid, smem, cluster, pdl, stream);
    return launch_one<DT, MODE, 1, 16>(p, grid, smem, cluster, pdl, stream);
  }
  if (r <= 16) return launch_one<DT, MODE, 8, 2>(p, grid, smem, cluster, pdl, stream);
  if (r <= 32) return launch_one<DT, MODE, 8, 4>(p, grid, smem, cluster, pdl, stream);
  if (r <= 64) return launch_one<DT, MODE, 8, 8>(p, grid, smem, cluster, pdl, stream);
  return launch_one<DT, MODE, 4, 16>(p, grid, smem, cluster, pdl, stream);
}

}  // namespace decode
}  // namespace mlora
