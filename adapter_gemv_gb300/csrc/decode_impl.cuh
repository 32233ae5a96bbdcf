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
//   * Every byte a CTA needs is requested into L2 at CTA start with bulk prefetches
//     (cp.async.bulk.prefetch.L2): HBM traffic begins at once, costs no shared memory, and
//     -- with programmatic dependent launch -- runs ahead of griddepcontrol.wait, overlapping
//     the previous kernel. The arithmetic then reads L2 with coalesced 16-byte loads; only a
//     block of x rows and the exchange buffers live in shared memory, so many CTAs fit per SM.
//   * Programmatic dependent launch (when the caller enables it): a kernel lets the next one in
//     the stream start at once.
//     Before griddepcontrol.wait a CTA only reads what no kernel of this library writes (the
//     rows' metadata, the pool, the page tables); x, y and v, which the previous kernel may
//     have written, are read after the wait (they may be prefetched into L2 before it).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace mlora {
namespace decode {

constexpr int NTHREADS = 256;
constexpr int NWARPS = NTHREADS / 32;
constexpr int SCAN_CAP = 1024;  // segment offsets staged per scan round
constexpr int MAX_CS = 16;      // CTAs per tile (cluster size)
constexpr int RANK_CACHE = 1024; // pools with at most this many slots: rank/scale read in the first round trip

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
__device__ void resolve_tile(const DecodeParams &p, const ProblemDev &pr, int t, TileInfo *ti, int32_t *scan,
                             int32_t *rank_c, float *scale_c) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool cached = pr.pool.num_slots <= RANK_CACHE;
  if (tid == 0) {
    ti->skip = 1;
    ti->bad = 0;
    ti->nr = 0;
  }
  if (cached) {  // loaded together with the row metadata: one round trip for the whole resolve
    for (int q = tid; q < pr.pool.num_slots; q += NTHREADS) {
      rank_c[q] = pr.pool.rank[q];
      scale_c[q] = pr.pool.scale[q];
    }
  }
  __syncthreads();
  if (p.seg_off != nullptr) {
    int32_t carry = 0, found = 0, bad = 0;
    for (int base = 0; base < p.nseg; base += SCAN_CAP) {
      const int cnt = min(SCAN_CAP, p.nseg - base);
      for (int q = tid; q <= cnt; q += NTHREADS) {
        scan[q] = p.seg_off[base + q];
        if (q < cnt) scan[SCAN_CAP + 1 + q] = p.seg_slot[base + q];  // one round trip for both
      }
      __syncthreads();
      if (warp == 0) {
        if (lane == 0 && ((base == 0 && scan[0] != 0) || (base + cnt == p.nseg && scan[cnt] != p.M))) bad = 1;
        for (int q0 = 0; q0 < cnt; q0 += 32) {
          const int q = q0 + lane;
          int32_t len = 0, lo = 0;
          if (q < cnt) {
            lo = scan[q];
            len = scan[q + 1] - lo;
            if (len < 0 || lo < 0 || scan[q + 1] > p.M) bad = 1;
            if (p.tc_min > 0 && len >= p.tc_min) len = 0;  // a tensor-core kernel does this segment
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
            ti->slot = scan[SCAN_CAP + 1 + q];
          }
          found |= __any_sync(0xffffffffu, mine);
          carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
          if (bad) {
            ti->bad = MLORA_STATUS_BAD_OFFSETS;
            found = 0;
          }
        }
      }
      if (base + SCAN_CAP < p.nseg) __syncthreads();  // the next round overwrites scan
    }
    if (p.nseg == 0 && tid == 0 && p.seg_off[0] != p.M) ti->bad = MLORA_STATUS_BAD_OFFSETS;
    if (tid == 0) ti->skip = (found && !ti->bad) ? 0 : 1;
  } else if (tid == 0 && t < p.M) {
    ti->row0 = t;
    ti->nr = 1;
    ti->slot = p.row_slot[t];
    ti->skip = 0;
  }  // (the BGMV slot load overlaps the rank/scale table loads above: both precede one barrier)
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
      rank = cached ? rank_c[s] : pl.rank[s];
      scale = cached ? scale_c[s] : pl.scale[s];
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
//   [0, 64)      mbarriers: xbar (exchange), bbar (B rows staged in shared memory)
//   [64, 96)     TileInfo
//   gbuf         [cs][RT][r_alloc] floats: every CTA's partial v (cluster modes)
//   vsm          [RT][r_alloc] floats: the summed v of the tile
//   scan         [2 * SCAN_CAP + 1] ints: segment offsets and slots while resolving the tile
//   rank_c/scale_c [RANK_CACHE] ints / floats: the pool's rank and scale tables (small pools)
//   xs           [RT][kb] elements: one pass of the tile's x rows (shrink)
//   bs           [r_alloc][nb] elements: this CTA's B rows, when staged (expand)
struct Layout {
  int gbuf, vsm, scan, rank_c, scale_c, xs, bs, total;
  __host__ __device__ static Layout make(int cs, int rt, int r_alloc, int kb, int nb_staged) {
    Layout L;
    L.gbuf = 128;
    L.vsm = L.gbuf + cs * rt * r_alloc * 4;
    L.scan = L.vsm + rt * r_alloc * 4;
    L.rank_c = L.scan + (2 * SCAN_CAP + 1) * 4;
    L.scale_c = L.rank_c + RANK_CACHE * 4;
    L.xs = (L.scale_c + RANK_CACHE * 4 + 127) & ~127;
    L.bs = (L.xs + rt * kb * 2 + 127) & ~127;
    L.total = L.bs + r_alloc * nb_staged * 2;
    return L;
  }
};

// A rows are read in passes of KB = 256 * UK elements of the CTA's K slice: lane l of warp w
// holds chunks c8 = l + 32u (u < UK) of rank rows j = w + 8jj (jj < JPW) -- JPW * UK = 16
// loads of 16 bytes in flight per thread, issued together.
template <int JPW>
struct Pass {
  static constexpr int UK = 16 / JPW;
  static constexpr int KB = 256 * UK;
};

template <int DT, int MODE, int RT, int JPW>
__global__ void __launch_bounds__(NTHREADS) decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int UK = Pass<JPW>::UK;
  constexpr int KB = Pass<JPW>::KB;
  const int cs = p.csplit;  // CTAs per tile: the cluster (SHRINK, FUSED) or the N-split (EXPAND)
  const bool stage_b = p.nb > 0;  // B rows of the CTA's slice go to shared memory before the wait
  const Layout L = Layout::make(MODE == MODE_EXPAND ? 1 : cs, RT, p.r_alloc, KB, p.nb);
  uint64_t *xbar = reinterpret_cast<uint64_t *>(smem);
  uint64_t *bbar = xbar + 1;
  TileInfo *ti = reinterpret_cast<TileInfo *>(smem + 64);
  float *gbuf = reinterpret_cast<float *>(smem + L.gbuf);
  float *vsm = reinterpret_cast<float *>(smem + L.vsm);
  int32_t *scan = reinterpret_cast<int32_t *>(smem + L.scan);
  int32_t *rank_c = reinterpret_cast<int32_t *>(smem + L.rank_c);
  float *scale_c = reinterpret_cast<float *>(smem + L.scale_c);
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem + L.xs);
  uint16_t *bs = reinterpret_cast<uint16_t *>(smem + L.bs);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool clustered = (MODE != MODE_EXPAND) && cs > 1;
  const uint32_t c = (MODE == MODE_EXPAND) ? (blockIdx.x % cs) : cluster_ctarank();
  const int64_t unit = blockIdx.x / cs;  // (problem, tile)
  const int prob = (int)(unit / p.tiles);
  const int t = (int)(unit % p.tiles);
  const ProblemDev &pr = p.prob[prob];
  const PoolDev &pl = pr.pool;

  if (tid == 0) {
    mbar_init(xbar, 1);
    mbar_init(bbar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (clustered) cluster_arrive_relaxed();  // peers may push into our gbuf once everyone arrived
  pdl_launch_dependents();                  // the next kernel may start; it waits for us before reading our outputs

  resolve_tile<MODE>(p, pr, t, ti, scan, rank_c, scale_c);
  if (c == 0 && tid == 0 && ti->bad) report(p.status, ti->bad);
  const bool active = !ti->skip;  // uniform across the block and across the cluster
  const int row0 = ti->row0, nr = ti->nr, s = ti->slot, rank = ti->rank;
  const float scale = ti->scale;

  // This CTA's slices of d_in and d_out.
  const int kchunk = ((pl.d_in + cs - 1) / cs + 7) & ~7;
  const int nchunk = ((pl.d_out + cs - 1) / cs + 7) & ~7;
  const int k_begin = min((int)c * kchunk, pl.d_in), k_end = min(k_begin + kchunk, pl.d_in);
  const int n_begin = min((int)c * nchunk, pl.d_out), n_end = min(n_begin + nchunk, pl.d_out);
  const bool do_shrink = MODE != MODE_EXPAND && active;
  const bool do_expand = MODE != MODE_SHRINK && active;
  const bool b_staged = do_expand && stage_b && n_end > n_begin;
  const uint64_t evict_first = policy_evict_first();

  // Everything that no kernel writes -- the adapter rows -- is requested before waiting for the
  // previous kernel: the first pass of A into registers, this CTA's B rows into shared memory.
  // The activation rows are prefetched into L2 (harmless: L2 is the point of coherence).
  if (active && warp == 0) {
    if (do_shrink && k_end > k_begin)
      for (int i = lane; i < nr; i += 32)
        prefetch_l2(pr.x + (int64_t)(row0 + i) * pr.ldx + k_begin, (uint32_t)(k_end - k_begin) * 2);
    if (do_expand && n_end > n_begin) {
      for (int i = lane; i < nr; i += 32)
        prefetch_l2(pr.y + (int64_t)(row0 + i) * pr.ldy + n_begin, (uint32_t)(n_end - n_begin) * 2);
      if (b_staged) {
        if (lane == 0) mbar_arrive_expect_tx(bbar, (uint32_t)(rank * (n_end - n_begin) * 2));
        __syncwarp();
        for (int j = lane; j < rank; j += 32)
          bulk_g2s_hint(bs + j * p.nb, b_row(pl, s, pr.layer, j) + n_begin, (uint32_t)(n_end - n_begin) * 2, bbar,
                        evict_first);
      } else {
        for (int j = lane; j < rank; j += 32)
          prefetch_l2(b_row(pl, s, pr.layer, j) + n_begin, (uint32_t)(n_end - n_begin) * 2);
      }
    }
    if (do_shrink && k_end - k_begin > KB)
      for (int j = lane; j < rank; j += 32)
        prefetch_l2(a_row(pl, s, pr.layer, j) + k_begin + KB, (uint32_t)(k_end - k_begin - KB) * 2);
    if (clustered && lane == 0) mbar_arrive_expect_tx(xbar, (uint32_t)(cs * nr * rank * 4));
  }
  // Prefetch hint: the adapter rows the next call will read for this tile's slot, shared out
  // over the nprob * cs CTAs of this tile (row items round-robin).
  if (active && p.nnext > 0 && warp == 1) {
    const int W = p.nprob * cs, w = prob * cs + (int)c;
    for (int q = 0; q < p.nnext; ++q) {
      const PoolDev &np = p.next_pool[q];
      if (s >= np.num_slots) continue;
      const int nrank = np.rank[s];
      if (nrank < 1 || nrank > np.r_max) continue;
      for (int item = lane; item < 2 * nrank; item += 32) {
        if ((q * 2 * nrank + item) % W != w) continue;
        const int j = item >> 1;
        const int64_t tix = ((int64_t)s * np.num_layers + p.next_layer[q]) * np.r_max + j;
        if (item & 1) {
          const int64_t pg = np.kind == MLORA_POOL_STACKED ? 0 : np.b_tab[tix];
          if (np.kind == MLORA_POOL_PAGED && (pg < 0 || pg >= np.num_pages)) continue;
          prefetch_l2(np.kind == MLORA_POOL_STACKED ? np.b + tix * np.d_out : np.pages + pg * np.page_elems,
                      (uint32_t)np.d_out * 2);
        } else {
          const int64_t pg = np.kind == MLORA_POOL_STACKED ? 0 : np.a_tab[tix];
          if (np.kind == MLORA_POOL_PAGED && (pg < 0 || pg >= np.num_pages)) continue;
          prefetch_l2(np.kind == MLORA_POOL_STACKED ? np.a_t + tix * np.d_in : np.pages + pg * np.page_elems,
                      (uint32_t)np.d_in * 2);
        }
      }
    }
  }

  uint4 a[JPW][UK];
  auto load_a = [&](int kb0) {
    const int n8 = min(KB, k_end - kb0) >> 3;
#pragma unroll
    for (int jj = 0; jj < JPW; ++jj) {
      const int j = warp + jj * NWARPS;
#pragma unroll
      for (int u = 0; u < UK; ++u) {
        const int c8 = lane + 32 * u;
        if (j < rank && c8 < n8) a[jj][u] = ldg_stream(a_row(pl, s, pr.layer, j) + kb0 + c8 * 8, evict_first);
      }
    }
  };
  if (do_shrink) load_a(k_begin);

  pdl_wait();  // the previous kernel in the stream has finished; its writes are visible

  // y of this thread's first YPRE column chunks (one-row tiles), requested now so it is here by
  // the expand
  constexpr int YPRE = 4;
  uint4 ypre[YPRE];
  if (RT == 1 && do_expand) {
    const int n8 = (n_end - n_begin) >> 3;
#pragma unroll
    for (int q = 0; q < YPRE; ++q)
      if (tid + q * NTHREADS < n8) ypre[q] = ldg_u4(pr.y + (int64_t)row0 * pr.ldy + n_begin + (tid + q * NTHREADS) * 8);
  }
  int timed_out = 0;

  // ---------------- shrink: partial v over this CTA's slice of d_in ----------------
  if (MODE != MODE_EXPAND) {
    float acc[RT][JPW];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) acc[i][jj] = 0.f;

    if (do_shrink) {
      for (int kb0 = k_begin; kb0 < k_end; kb0 += KB) {
        const int n8 = min(KB, k_end - kb0) >> 3;
        if (kb0 != k_begin) load_a(kb0);
        // x rows of this pass -> shared memory (read by every warp)
        for (int e = tid; e < nr * n8; e += NTHREADS) {
          const int i = e / n8, c8 = e % n8;
          *reinterpret_cast<uint4 *>(xs + i * KB + c8 * 8) = ldg_u4(pr.x + (int64_t)(row0 + i) * pr.ldx + kb0 + c8 * 8);
        }
        __syncthreads();
#pragma unroll
        for (int jj = 0; jj < JPW; ++jj) {
          const int j = warp + jj * NWARPS;
          if (j < rank) {
#pragma unroll
            for (int u = 0; u < UK; ++u) {
              const int c8 = lane + 32 * u;
              if (c8 < n8) {
                float af[8];
                unpack8<DT>(a[jj][u], af);
#pragma unroll
                for (int i = 0; i < RT; ++i) {
                  if (i < nr) {
                    float xf[8];
                    unpack8<DT>(*reinterpret_cast<const uint4 *>(xs + i * KB + c8 * 8), xf);
                    float sacc = acc[i][jj];
#pragma unroll
                    for (int e = 0; e < 8; ++e) sacc = fmaf(xf[e], af[e], sacc);
                    acc[i][jj] = sacc;
                  }
                }
              }
            }
          }
        }
        __syncthreads();  // xs is rewritten by the next pass
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
      cluster_wait();  // every peer has initialised its exchange barrier
      if (do_shrink && lane < cs) {
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
      if (do_shrink) {
        const int ok = mbar_wait_cluster(xbar, 0) ? 1 : 0;
        timed_out = __syncthreads_or(!ok);
        if (!timed_out) {
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
      }
    } else if (do_shrink && lane == 0) {
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
  if (b_staged && !timed_out) {
    const int ok = mbar_wait(bbar, 0) ? 1 : 0;
    timed_out = __syncthreads_or(!ok);
  }
  if (do_expand && !timed_out) {
    const int n8 = (n_end - n_begin) >> 3;
    for (int c8 = tid; c8 < n8; c8 += NTHREADS) {
      const int n0 = n_begin + c8 * 8;
      float acc[RT][8];
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
      if (b_staged) {
        for (int j = 0; j < rank; ++j) {
          float bf[8];
          unpack8<DT>(*reinterpret_cast<const uint4 *>(bs + j * p.nb + c8 * 8), bf);
#pragma unroll
          for (int i = 0; i < RT; ++i) {
            if (i < nr) {
              const float vij = vsm[i * p.r_alloc + j];
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(vij, bf[e], acc[i][e]);
            }
          }
        }
      } else {
        constexpr int UB = RT == 1 ? 16 : 4;  // B loads in flight per thread
        for (int j0 = 0; j0 < rank; j0 += UB) {
          uint4 b[UB];
#pragma unroll
          for (int u = 0; u < UB; ++u)
            if (j0 + u < rank) b[u] = ldg_stream(b_row(pl, s, pr.layer, j0 + u) + n0, evict_first);
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            if (j0 + u < rank) {
              float bf[8];
              unpack8<DT>(b[u], bf);
#pragma unroll
              for (int i = 0; i < RT; ++i) {
                if (i < nr) {
                  const float vij = vsm[i * p.r_alloc + j0 + u];
#pragma unroll
                  for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(vij, bf[e], acc[i][e]);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RT; ++i) {
        if (i < nr) {
          float yf[8];
          const int q = (c8 - tid) / NTHREADS;
          uint4 yw;
          if (RT == 1 && q < YPRE) {
#pragma unroll
            for (int qq = 0; qq < YPRE; ++qq)
              if (qq == q) yw = ypre[qq];
          } else {
            yw = ldg_u4(pr.y + (int64_t)(row0 + i) * pr.ldy + n0);
          }
          unpack8<DT>(yw, yf);
#pragma unroll
          for (int e = 0; e < 8; ++e) yf[e] = fmaf(scale, acc[i][e], yf[e]);
          *reinterpret_cast<uint4 *>(pr.y + (int64_t)(row0 + i) * pr.ldy + n0) = pack8<DT>(yf);
        }
      }
    }
  }

  if (b_staged && timed_out) (void)mbar_wait(bbar, 0, 100000000ull);  // copies in flight land before exit
  if (timed_out && tid == 0) report(p.status, MLORA_STATUS_TIMEOUT);
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
