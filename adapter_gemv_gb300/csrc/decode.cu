// decode.cu -- CUDA-core kernels for decode-sized row tiles (sm_103a).
//
// Work unit: a TILE = up to RT consecutive rows that use one adapter (a piece of an SGMV
// segment, or one BGMV row). The delta of a tile is a handful of dot products over d_in
// (shrink) and a handful of axpys over d_out (expand): matrix-vector work that is bound by
// HBM bandwidth, so it runs on the CUDA cores (Punica section 3.4, "The degenerate case":
// the one-request-per-adapter schedule uses coalesced CUDA-core loads, not tensor cores).
//
// GB300 design:
//   * Split-K shrink (Punica section 3.4, "SGMV-shrink schedule") across the CTAs of a
//     thread-block CLUSTER. Each CTA reduces its slice of d_in into partial v in shared
//     memory; the partials are summed through distributed shared memory after a hardware
//     cluster barrier. No grid-wide barrier, no workspace, no atomics, fixed summation order.
//   * Output-split expand (Punica section 3.4, "SGMV-expand schedule"): each CTA owns a slice
//     of d_out, streams B[s] rows for that slice once per tile and rewrites y in place.
//   * FUSED mode does both in one launch: the cluster reduces v on chip, then each CTA
//     expands its d_out slice. B and y of the slice are requested at kernel start, so their
//     HBM latency overlaps the shrink.
//   * Operands move with the TMA engine's bulk copies (cp.async.bulk) into a shared-memory
//     ring whose stages complete on mbarriers; one warp issues them, all warps compute.
//   * Adapter rows come from a stacked pool or, through page tables, from a paged pool
//     (S-LoRA "Unified Paging"): every rank-row is one contiguous run, so both gather the same
//     way.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace mlora {

namespace {

constexpr int NTHREADS = 256;
constexpr int NWARPS = NTHREADS / 32;
constexpr int MAX_STAGES = 4;
constexpr int SCAN_CAP = 2048;  // offsets staged per scan round (ints)

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

// Resolve virtual tile `t` of problem `pr` into `ti` (whole block participates).
// SGMV: segments contribute ceil(len / rt) tiles each, in segment order.
// BGMV: tile t is row t.
template <int MODE>
__device__ void resolve_tile(const DecodeParams &p, const ProblemDev &pr, int t, TileInfo *ti, int32_t *scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();  // every thread is done with the previous tile's info and scan buffer
  if (tid == 0) {
    ti->skip = 1;
    ti->bad = 0;
    ti->nr = 0;
  }
  __syncthreads();
  if (p.seg_off != nullptr) {
    // The block stages the offsets in shared memory; warp 0 walks them with a prefix sum of
    // tiles per segment. Runs once per tile; the offsets are L2-resident after the first CTA.
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
          if (!found && q < cnt && t >= excl && t < excl + nt) {
            const int32_t sub = t - excl;
            ti->row0 = lo + sub * p.rt;
            ti->nr = min(p.rt, len - sub * p.rt);
            ti->slot = p.seg_slot[base + q];
          }
          found |= __any_sync(0xffffffffu, q < cnt && t >= excl && t < excl + nt);
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
        ti->nr = 0;
        found = 0;
      }
      ti->skip = found ? 0 : 1;
    }
  } else {
    if (tid == 0 && t < p.M) {
      ti->row0 = t;
      ti->nr = 1;
      ti->slot = p.row_slot[t];
      ti->skip = 0;
    }
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

template <int DT, int MODE, int RT, int JPW>
__global__ void __launch_bounds__(NTHREADS) decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full_k = reinterpret_cast<uint64_t *>(smem);
  uint64_t *full_e = full_k + MAX_STAGES;
  TileInfo *ti = reinterpret_cast<TileInfo *>(smem + 2 * MAX_STAGES * sizeof(uint64_t));
  float *partial = reinterpret_cast<float *>(smem + 128);
  float *vsm = partial + RT * p.r_alloc;
  uint8_t *ring_k = smem + 128 + 2 * RT * p.r_alloc * (int)sizeof(float);
  ring_k = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ring_k) + 127) & ~uintptr_t(127));
  const int stage_k_bytes = (p.r_alloc + RT) * p.kb * 2;
  const int stage_e_bytes = (p.r_alloc + RT) * p.nb * 2;
  uint8_t *ring_e = ring_k + p.sk * stage_k_bytes;
  int32_t *scan = reinterpret_cast<int32_t *>(ring_e + p.se * stage_e_bytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const ProblemDev &pr = p.prob[blockIdx.z];
  const PoolDev &pl = pr.pool;
  const uint32_t c = (MODE == MODE_EXPAND) ? blockIdx.x : cluster_ctarank();
  const int csplit = (MODE == MODE_EXPAND) ? (int)gridDim.x : p.csplit;

  if (tid == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&full_e[s], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // K and N ranges of this CTA.
  const int kchunk = ((pl.d_in + csplit - 1) / csplit + 7) & ~7;
  const int nchunk = ((pl.d_out + csplit - 1) / csplit + 7) & ~7;
  const int k_begin = min((int)c * kchunk, pl.d_in), k_end = min(k_begin + kchunk, pl.d_in);
  const int n_begin = min((int)c * nchunk, pl.d_out), n_end = min(n_begin + nchunk, pl.d_out);
  const int nkb = (MODE == MODE_EXPAND) ? 0 : (k_end - k_begin + p.kb - 1) / p.kb;
  const int nnb = (MODE == MODE_SHRINK) ? 0 : (n_end - n_begin + p.nb - 1) / p.nb;
  const uint64_t evict_first = policy_evict_first();

  // Ring bookkeeping: blocks issued and consumed so far (stage = g % stages, parity = g / stages).
  uint32_t gk = 0, ge = 0, issued_k = 0, issued_e = 0;
  // Block-uniform: once a bounded wait gives up, this CTA stops issuing, computing and
  // writing, but keeps taking part in every cluster barrier so its peers cannot hang.
  int timed_out = 0;

  for (int t = blockIdx.y; t < p.tiles; t += gridDim.y) {
    resolve_tile<MODE>(p, pr, t, ti, scan);
    if (c == 0 && tid == 0 && ti->bad) report(p.status, ti->bad);
    if (ti->skip) continue;  // uniform across the block and across the cluster
    const int row0 = ti->row0, nr = ti->nr, s = ti->slot, rank = ti->rank;
    const float scale = ti->scale;

    // Producer: warp 0 issues one block (rank adapter rows + nr activation rows) per stage.
    auto issue_k = [&](int blk) {
      const uint32_t g = gk + blk;
      const int stage = g % p.sk;
      const int k0 = k_begin + blk * p.kb, kv = min(p.kb, k_end - k0);
      uint8_t *base = ring_k + stage * stage_k_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&full_k[stage], (uint32_t)((rank + nr) * kv * 2));
      __syncwarp();
      for (int q = lane; q < rank + nr; q += 32) {
        if (q < rank) {
          bulk_g2s_hint(base + q * p.kb * 2, a_row(pl, s, pr.layer, q) + k0, kv * 2, &full_k[stage], evict_first);
        } else {
          const int i = q - rank;
          bulk_g2s(base + (p.r_alloc + i) * p.kb * 2, pr.x + (int64_t)(row0 + i) * pr.ldx + k0, kv * 2,
                   &full_k[stage]);
        }
      }
    };
    auto issue_e = [&](int blk) {
      const uint32_t g = ge + blk;
      const int stage = g % p.se;
      const int n0 = n_begin + blk * p.nb, nv = min(p.nb, n_end - n0);
      uint8_t *base = ring_e + stage * stage_e_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&full_e[stage], (uint32_t)((rank + nr) * nv * 2));
      __syncwarp();
      for (int q = lane; q < rank + nr; q += 32) {
        if (q < rank) {
          bulk_g2s_hint(base + q * p.nb * 2, b_row(pl, s, pr.layer, q) + n0, nv * 2, &full_e[stage], evict_first);
        } else {
          const int i = q - rank;
          bulk_g2s(base + (p.r_alloc + i) * p.nb * 2, pr.y + (int64_t)(row0 + i) * pr.ldy + n0, nv * 2,
                   &full_e[stage]);
        }
      }
    };
    if (!timed_out) {
      const int pk = min(nkb, p.sk), pe = min(nnb, p.se);
      if (warp == 0) {
        for (int b = 0; b < pk; ++b) issue_k(b);
        for (int b = 0; b < pe; ++b) issue_e(b);
      }
      issued_k = gk + pk;
      issued_e = ge + pe;
    }

    // ---------------- shrink: partial v over this CTA's slice of d_in ----------------
    if (MODE != MODE_EXPAND) {
      float acc[RT][JPW];
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int jj = 0; jj < JPW; ++jj) acc[i][jj] = 0.f;

      int done = 0;
      for (int blk = 0; blk < nkb && !timed_out; ++blk) {
        const uint32_t g = gk + blk;
        const int stage = g % p.sk;
        const int ok = mbar_wait(&full_k[stage], (g / p.sk) & 1u) ? 1 : 0;
        timed_out = __syncthreads_or(!ok);
        if (timed_out) break;
        ++done;
        const int kv = min(p.kb, k_end - (k_begin + blk * p.kb));
        const uint16_t *As = reinterpret_cast<const uint16_t *>(ring_k + stage * stage_k_bytes);
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
        if (warp == 0 && blk + p.sk < nkb) issue_k(blk + p.sk);
        if (blk + p.sk < nkb) issued_k = gk + blk + p.sk + 1;
      }
      gk += done;

      // warp-level reduction of each (row, rank) dot product; lane 0 writes the partial
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) {
        const int j = warp + jj * NWARPS;
        if (j < rank) {
#pragma unroll
          for (int i = 0; i < RT; ++i) {
            if (i < nr) {
              float sv = acc[i][jj];
#pragma unroll
              for (int d = 16; d > 0; d >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, d);
              if (lane == 0) partial[i * p.r_alloc + j] = sv;
            }
          }
        }
      }
      __syncthreads();

      // split-K combine over the cluster, in CTA-rank order (deterministic)
      const int nent = nr * rank;
      if (csplit > 1) cluster_sync();
      for (int e = tid; e < nent; e += NTHREADS) {
        if (MODE == MODE_SHRINK && e % csplit != (int)c) continue;
        const int i = e / rank, j = e % rank;
        float sum = 0.f;
        if (csplit > 1) {
          for (int q = 0; q < csplit; ++q) sum += dsmem_ld_f32(dsmem_addr(&partial[i * p.r_alloc + j], q));
        } else {
          sum = partial[i * p.r_alloc + j];
        }
        if (MODE == MODE_SHRINK) {
          if (!timed_out) pr.v[(int64_t)(row0 + i) * pl.r_max + j] = sum;
        } else {
          vsm[i * p.r_alloc + j] = sum;
        }
      }
      if (csplit > 1) cluster_sync();  // partials may be reused / released only after every read
      else __syncthreads();
    } else {
      // expand only: v rows of this tile from global memory
      for (int e = tid; e < nr * rank; e += NTHREADS) {
        const int i = e / rank, j = e % rank;
        vsm[i * p.r_alloc + j] = pr.v[(int64_t)(row0 + i) * pl.r_max + j];
      }
      __syncthreads();
    }

    // ---------------- expand: y[rows][this CTA's slice of d_out] ----------------
    if (MODE != MODE_SHRINK) {
      int done = 0;
      for (int blk = 0; blk < nnb && !timed_out; ++blk) {
        const uint32_t g = ge + blk;
        const int stage = g % p.se;
        const int ok = mbar_wait(&full_e[stage], (g / p.se) & 1u) ? 1 : 0;
        timed_out = __syncthreads_or(!ok);
        if (timed_out) break;
        ++done;
        const int n0 = n_begin + blk * p.nb, nv = min(p.nb, n_end - n0);
        const uint16_t *Bs = reinterpret_cast<const uint16_t *>(ring_e + stage * stage_e_bytes);
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
        if (warp == 0 && blk + p.se < nnb) issue_e(blk + p.se);
        if (blk + p.se < nnb) issued_e = ge + blk + p.se + 1;
      }
      ge += done;
    }
  }
  if (timed_out) {
    // Wait (bounded) for this CTA's copies still in flight before its shared memory goes away.
    for (uint32_t g = gk; g < issued_k; ++g) (void)mbar_wait(&full_k[g % p.sk], (g / p.sk) & 1u, 100000000ull);
    for (uint32_t g = ge; g < issued_e; ++g) (void)mbar_wait(&full_e[g % p.se], (g / p.se) & 1u, 100000000ull);
    if (tid == 0) report(p.status, MLORA_STATUS_TIMEOUT);
  }
}

template <int DT, int MODE, int RT, int JPW>
cudaError_t launch_one(const DecodeParams &p, dim3 grid, size_t smem, int cluster, cudaStream_t stream) {
  auto kern = decode_kernel<DT, MODE, RT, JPW>;
  static int configured_smem[64] = {0};  // per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured_smem[dev] < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (cluster > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    configured_smem[dev] = (int)smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (MODE != MODE_EXPAND) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int DT, int MODE>
cudaError_t dispatch_rt(const DecodeParams &p, dim3 grid, size_t smem, int cluster, cudaStream_t stream, int rt) {
  if (rt == 8) return launch_one<DT, MODE, 8, 8>(p, grid, smem, cluster, stream);
  return launch_one<DT, MODE, 4, 16>(p, grid, smem, cluster, stream);
}

}  // namespace

// Host: choose the split, the stage sizes and the grid; launch.
cudaError_t launch_decode(int mode, int dtype, DecodeParams p, cudaStream_t stream, int force_csplit) {
  int r_alloc = 1, d_in_max = 8, d_out_max = 8;
  for (int q = 0; q < p.nprob; ++q) {
    r_alloc = max(r_alloc, p.prob[q].pool.r_max);
    d_in_max = max(d_in_max, p.prob[q].pool.d_in);
    d_out_max = max(d_out_max, p.prob[q].pool.d_out);
  }
  const int RT = (r_alloc <= 64) ? 8 : 4;
  p.r_alloc = r_alloc;
  p.rt = (p.seg_off != nullptr) ? RT : 1;
  const int64_t tiles = (p.seg_off != nullptr) ? (int64_t)p.nseg + (p.M + p.rt - 1) / p.rt : (int64_t)p.M;
  if (tiles <= 0) return cudaSuccess;
  p.tiles = (int32_t)tiles;

  const int stage_cap = 48 * 1024;
  const int row_bytes_cap = stage_cap / ((r_alloc + RT) * 2);  // elements per row per stage
  auto balanced = [&](int chunk) {
    const int cap = max(8, row_bytes_cap & ~7);
    const int nblk = (chunk + cap - 1) / cap;
    return (((chunk + nblk - 1) / nblk) + 7) & ~7;
  };
  int csplit;
  if (mode == MODE_EXPAND) {
    csplit = force_csplit > 0 ? force_csplit : max(1, (d_out_max + 511) / 512);
  } else {
    csplit = force_csplit > 0 ? force_csplit : min(8, max(1, (d_in_max + 511) / 512));
  }
  p.csplit = csplit;
  const int kchunk = ((d_in_max + csplit - 1) / csplit + 7) & ~7;
  const int nchunk = ((d_out_max + csplit - 1) / csplit + 7) & ~7;
  p.kb = (mode == MODE_EXPAND) ? 8 : balanced(kchunk);
  p.nb = (mode == MODE_SHRINK) ? 8 : balanced(nchunk);
  p.sk = (mode == MODE_EXPAND) ? 0 : min(MAX_STAGES, max(1, (kchunk + p.kb - 1) / p.kb));
  p.se = (mode == MODE_SHRINK) ? 0 : min(MAX_STAGES, max(1, (nchunk + p.nb - 1) / p.nb));
  // the scan buffer shares nothing with the rings (it is read while copies are in flight)
  size_t smem = 128 + 2 * (size_t)RT * r_alloc * sizeof(float) + 128;
  smem += (size_t)p.sk * (r_alloc + RT) * p.kb * 2 + (size_t)p.se * (r_alloc + RT) * p.nb * 2;
  smem += (SCAN_CAP + 1) * sizeof(int32_t);
  while (smem > 227 * 1024 && (p.sk > 1 || p.se > 1)) {
    if (p.sk >= p.se && p.sk > 1) {
      smem -= (size_t)(r_alloc + RT) * p.kb * 2;
      --p.sk;
    } else {
      smem -= (size_t)(r_alloc + RT) * p.nb * 2;
      --p.se;
    }
  }
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;

  dim3 grid(csplit, (unsigned)(tiles < 65535 ? tiles : 65535), p.nprob);
  const int cluster = (mode == MODE_EXPAND) ? 1 : csplit;
  const bool bf = dtype == MLORA_BF16;
  switch (mode) {
    case MODE_SHRINK:
      return bf ? dispatch_rt<MLORA_BF16, MODE_SHRINK>(p, grid, smem, cluster, stream, RT)
                : dispatch_rt<MLORA_FP16, MODE_SHRINK>(p, grid, smem, cluster, stream, RT);
    case MODE_EXPAND:
      return bf ? dispatch_rt<MLORA_BF16, MODE_EXPAND>(p, grid, smem, cluster, stream, RT)
                : dispatch_rt<MLORA_FP16, MODE_EXPAND>(p, grid, smem, cluster, stream, RT);
    default:
      return bf ? dispatch_rt<MLORA_BF16, MODE_FUSED>(p, grid, smem, cluster, stream, RT)
                : dispatch_rt<MLORA_FP16, MODE_FUSED>(p, grid, smem, cluster, stream, RT);
  }
}

}  // namespace mlora
