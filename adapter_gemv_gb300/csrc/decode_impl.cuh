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
//   * Staging. Before griddepcontrol.wait a CTA resolves its tile (one round trip for the row
//     metadata and the pool's rank table), loads its first pass of A rows into registers (zero
//     outside the slice and the rank) and bulk-copies its B rows into shared memory, over the
//     area the resolve used: the adapter rows stream in while the previous kernel runs. After
//     the wait one thread bulk-copies the tile's x rows (and y rows, when they fit) into shared
//     memory. Later passes of A, and B rows that do not fit, come from L2, prefetched there.
//   * Arithmetic runs on data already on chip, as straight-line code without per-chunk or
//     per-row guards (the staged operands are zero where they lie outside the tile). The shrink
//     meets packed 16-bit x and A directly in mixed-precision FMAs (fp32 sums, no unpacking);
//     the expand, whose v is fp32, uses the paired fp32 FMA.
//   * Programmatic dependent launch (when the caller enables it): a kernel lets the next one in
//     the stream start at once. Before griddepcontrol.wait a CTA only reads what no kernel of
//     this library writes (the rows' metadata, the pool, the page tables); x, y and v, which the
//     previous kernel may have written, are read after the wait (they may be prefetched into L2
//     before it).
//   * One cluster barrier phase only: every CTA arrives at start and waits before pushing (so
//     every peer's exchange barrier is initialised). No barrier at exit: a CTA leaves once its
//     own exchange barrier has counted every push into its shared memory, without waiting for
//     its peers' expand, and frees its SM for the next launch sooner.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

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
  // paged pools: the page-table rows of the tile's slot and layer (entry j * ppv + q = page of
  // piece q of vector j), A and B: the copy in shared memory when it fits, else the pool's tables.
  // Read from here at each use (kept out of the registers of the hot loops).
  const int32_t *a_tr, *b_tr;
};
static_assert(sizeof(TileInfo) <= 56, "TileInfo sits in [64, 120) of shared memory");

// Element k of row j of A^T (d_in elements) or of B (d_out elements) of slot s, layer `layer`.
// A paged vector spans ppv consecutive page-table entries: element k sits in entry
// k / page_elems at offset k % page_elems (a chunk of 8 elements never straddles two pages:
// page_elems is a multiple of 8). Square pages (ppv == 1) take one table entry per vector.
// Page of element k (k < 2^31) of a multi-page vector: k / page_elems by one multiply-high and a
// shift with the host's pe_mul / pe_shift (T. Granlund and P. Montgomery, "Division by Invariant
// Integers using Multiplication", 1994: q = (mulhi(m, k) + k) >> l, l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1).
__device__ __forceinline__ int page_of(const PoolDev &pl, int k) {
  return (int)((__umulhi((uint32_t)k, pl.pe_mul) + (uint32_t)k) >> pl.pe_shift);
}

// Branch-free, so that a batch of such addresses issues its table loads together (for one-page
// vectors q is 0). `tr` is the page-table row block of the tile's slot and layer: entry
// j * ppv + q holds the page of piece q of vector j (the tile's copy in shared memory, or the
// pool's table in global memory).
__device__ __forceinline__ const uint16_t *paged_elem(const PoolDev &pl, const int32_t *tr, int ppv, int j, int k) {
  const int q = page_of(pl, k);
  return pl.pages + (int64_t)tr[j * ppv + q] * pl.page_elems + (k - q * (int)pl.page_elems);
}

__device__ __forceinline__ const uint16_t *a_elem(const PoolDev &pl, int s, int layer, int j, int k,
                                                  const int32_t *a_tr) {
  if (pl.kind == MLORA_POOL_STACKED) return pl.a_t + (((int64_t)s * pl.num_layers + layer) * pl.r_max + j) * pl.d_in + k;
  return paged_elem(pl, a_tr, pl.a_ppv, j, k);
}

__device__ __forceinline__ const uint16_t *b_elem(const PoolDev &pl, int s, int layer, int j, int n,
                                                  const int32_t *b_tr) {
  if (pl.kind == MLORA_POOL_STACKED) return pl.b + (((int64_t)s * pl.num_layers + layer) * pl.r_max + j) * pl.d_out + n;
  return paged_elem(pl, b_tr, pl.b_ppv, j, n);
}

// Element n of the B rows of one slot and layer, for a batch of rank rows: the slot/layer part of
// the address and n's page are worked out once; row j then costs a multiply-add (and, paged, one
// page-table read).
struct BRows {
  const uint16_t *base;  // stacked: &B[s][layer][0][n]; paged: the pool
  const int32_t *tab;    // paged: the page-table entry of row 0's piece that holds n
  int64_t stride;        // stacked: d_out; paged: page_elems
  int32_t ppv, off;      // paged: table entries per row, n's offset in its page
  bool paged;
  __device__ __forceinline__ BRows(const PoolDev &pl, int s, int layer, int n, const int32_t *b_tr) {
    paged = pl.kind != MLORA_POOL_STACKED;
    if (!paged) {
      base = pl.b + ((int64_t)s * pl.num_layers + layer) * pl.r_max * pl.d_out + n;
      stride = pl.d_out;
      tab = nullptr;
      ppv = off = 0;
    } else {
      const int q = page_of(pl, n);
      base = pl.pages;
      stride = pl.page_elems;
      ppv = pl.b_ppv;
      tab = b_tr + q;
      off = n - q * (int)pl.page_elems;
    }
  }
  __device__ __forceinline__ const uint16_t *operator()(int j) const {
    return paged ? base + (int64_t)tab[j * ppv] * stride + off : base + (int64_t)j * stride;
  }
};

// f(ptr, off, count) for each piece of elements [k0, k1) of a vector that lies in one page (the
// whole range for a stacked pool or square pages); off is the piece's first element minus k0.
template <bool IS_A, class F>
__device__ __forceinline__ void vec_pieces(const PoolDev &pl, int s, int layer, int j, int k0, int k1,
                                           const int32_t *tr, F f) {
  const int ppv = IS_A ? pl.a_ppv : pl.b_ppv;
  if (pl.kind == MLORA_POOL_STACKED || ppv == 1) {
    if (k1 > k0) f(IS_A ? a_elem(pl, s, layer, j, k0, tr) : b_elem(pl, s, layer, j, k0, tr), 0, k1 - k0);
    return;
  }
  const int pe = (int)pl.page_elems;
#pragma unroll 1
  for (int k = k0; k < k1;) {
    const int end = min(k1, (page_of(pl, k) + 1) * pe);
    f(IS_A ? a_elem(pl, s, layer, j, k, tr) : b_elem(pl, s, layer, j, k, tr), k - k0, end - k);
    k = end;
  }
}

// Resolve virtual tile `t` of problem `pr` into `ti` (whole block participates; reads only
// metadata that no kernel of this library writes).
// SGMV: segments contribute ceil(len / rt) tiles each, in segment order. BGMV: tile t is row t.
// Every metadata load of the first scan round (offsets, slots, the pool's rank and scale tables
// when it has at most RANK_CACHE slots) is in flight at once: one round trip to memory.
template <int MODE>
__device__ void resolve_tile(const DecodeParams &p, const ProblemDev &pr, int t, TileInfo *ti, int32_t *scan,
                             int32_t *rank_c, float *scale_c, int32_t *ptab) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool cached = pr.pool.num_slots <= RANK_CACHE;
  const bool sgmv = p.seg_off != nullptr;
  const int cnt0 = sgmv ? min(SCAN_CAP, p.nseg) : 0;
  constexpr int RC = RANK_CACHE / NTHREADS;
  constexpr int SC = (SCAN_CAP + 1 + NTHREADS - 1) / NTHREADS;
  int32_t rk[RC], so[SC], ss[SC];
  float sc[RC];
  int32_t row_slot = 0, row_t = t;
#pragma unroll
  for (int i = 0; i < RC; ++i) {
    const int q = tid + i * NTHREADS;
    if (cached && q < pr.pool.num_slots) {
      rk[i] = pr.pool.rank[q];
      sc[i] = pr.pool.scale[q];
    }
  }
#pragma unroll
  for (int i = 0; i < SC; ++i) {
    const int q = tid + i * NTHREADS;
    if (sgmv && q <= cnt0) so[i] = p.seg_off[q];
    if (sgmv && q < cnt0) ss[i] = p.seg_slot[q];
  }
  if (!sgmv && tid == 0 && t < p.M) {
    if (p.perm) {  // grouped order: tile t is row perm[t]
      row_t = p.perm[t];
      row_slot = p.sslot[t];
    } else {
      row_slot = p.row_slot[t];
    }
  }
#pragma unroll
  for (int i = 0; i < RC; ++i) {
    const int q = tid + i * NTHREADS;
    if (cached && q < pr.pool.num_slots) {
      rank_c[q] = rk[i];
      scale_c[q] = sc[i];
    }
  }
#pragma unroll
  for (int i = 0; i < SC; ++i) {
    const int q = tid + i * NTHREADS;
    if (sgmv && q <= cnt0) scan[q] = so[i];
    if (sgmv && q < cnt0) scan[SCAN_CAP + 1 + q] = ss[i];
  }
  if (tid == 0) {
    ti->skip = 1;
    ti->bad = 0;
    ti->nr = 0;
  }
  __syncthreads();
  if (sgmv && p.rt == 1 && pr.tc_min == 0 && p.nseg <= SCAN_CAP) {
    // One-row tiles, every segment here: tile t is row t, in the segment whose offset is the last
    // one <= t (one ballot per 32 offsets); the offsets are checked the same way.
    if (warp == 0) {
      const int cnt = p.nseg;
      int le = 0, bad = 0;
      for (int q0 = 0; q0 <= cnt; q0 += 32) {
        const int q = q0 + lane;
        const int32_t o = q <= cnt ? scan[q] : 0;
        if (q < cnt) {
          const int32_t o1 = scan[q + 1];
          bad |= (o1 < o) | (o < 0) | (o1 > p.M);
        }
        le += __popc(__ballot_sync(0xffffffffu, q <= cnt && o <= t));
      }
      bad = __any_sync(0xffffffffu, bad) || scan[0] != 0 || scan[cnt] != p.M;
      if (lane == 0) {
        if (bad) {
          ti->bad = MLORA_STATUS_BAD_OFFSETS;
        } else if (t < p.M && le >= 1 && le <= cnt) {
          ti->row0 = t;
          ti->nr = 1;
          ti->slot = scan[SCAN_CAP + 1 + le - 1];
          ti->skip = 0;
        }
      }
    }
  } else if (sgmv) {
    int32_t carry = 0, found = 0, bad = 0;
    for (int base = 0; base < p.nseg; base += SCAN_CAP) {
      const int cnt = min(SCAN_CAP, p.nseg - base);
      if (base > 0) {  // later rounds (more than SCAN_CAP segments): load, then scan
        for (int q = tid; q <= cnt; q += NTHREADS) {
          scan[q] = p.seg_off[base + q];
          if (q < cnt) scan[SCAN_CAP + 1 + q] = p.seg_slot[base + q];
        }
        __syncthreads();
      }
      if (warp == 0) {
        if (lane == 0 && ((base == 0 && scan[0] != 0) || (base + cnt == p.nseg && scan[cnt] != p.M))) bad = 1;
        for (int q0 = 0; q0 < cnt; q0 += 32) {
          const int q = q0 + lane;
          int32_t len = 0, lo = 0;
          if (q < cnt) {
            lo = scan[q];
            len = scan[q + 1] - lo;
            if (len < 0 || lo < 0 || scan[q + 1] > p.M) bad = 1;
            if (pr.tc_min > 0 && len >= pr.tc_min) len = 0;  // a tensor-core kernel does this segment
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
        if (lane == 0 && bad) {
          ti->bad = MLORA_STATUS_BAD_OFFSETS;
          found = 0;
        }
      }
      if (base + SCAN_CAP < p.nseg) __syncthreads();  // the next round overwrites scan
    }
    if (p.nseg == 0 && tid == 0 && scan[0] != p.M) ti->bad = MLORA_STATUS_BAD_OFFSETS;
    if (tid == 0) ti->skip = (found && !ti->bad) ? 0 : 1;
  } else if (tid == 0 && t < p.M) {
    ti->row0 = row_t;
    ti->nr = 1;
    ti->slot = row_slot;
    ti->skip = 0;
  }
  // Adapter checks (warp 0, which wrote the tile above): slot range, rank range, page ids of
  // the rank-rows this mode reads.
  if (warp == 0) {
    __syncwarp();
    if (!ti->skip) {
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
          // every page of every vector j < rank this mode reads: entries [0, na) of the A table's
          // rows, then [na, na + nb) of the B table's, four loads in flight per lane at a time;
          // kept in shared memory (ptab, the same order) when they fit p.npt entries
          const int na = MODE != MODE_EXPAND ? rank * pl.a_ppv : 0;
          const int nt = na + (MODE != MODE_SHRINK ? rank * pl.b_ppv : 0);
          const bool keep = nt <= p.npt;
          for (int e0 = lane; e0 < nt; e0 += 128) {
            int32_t pg[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int e = e0 + 32 * u;
              pg[u] = e >= nt ? 0 : e < na ? pl.a_tab[t0 * pl.a_ppv + e] : pl.b_tab[t0 * pl.b_ppv + (e - na)];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int e = e0 + 32 * u;
              badp |= (pg[u] < 0 || pg[u] >= pl.num_pages);
              if (keep && e < nt) ptab[e] = pg[u];
            }
          }
          if (__any_sync(0xffffffffu, badp)) bad = MLORA_STATUS_BAD_PAGE;
          if (lane == 0) {
            ti->a_tr = keep ? ptab : pl.a_tab + t0 * pl.a_ppv;
            ti->b_tr = keep ? ptab + na : pl.b_tab + t0 * pl.b_ppv;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        ti->rank = rank;
        ti->scale = scale;
        ti->bad |= bad;
        ti->skip = (skip || bad) ? 1 : 0;
      }
    }
  }
  // The scan and table area is reused for staged B rows, written by bulk copies (the async
  // proxy): order this thread's accesses to it before them.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
}

// Shared-memory layout (dynamic):
//   [0, 64)      mbarriers: xbar (exchange), bbar (B rows staged), ibar (x slice), ybar (y slice)
//   [64, 120)    TileInfo; [120, 124) the short-tile count of a launch after tensor-core kernels
//   gbuf         [cs][RT][r_alloc] floats: every CTA's partial v (cluster modes)
//   vsm          [RT][r_alloc] floats: the summed v of the tile
//   xs           [RT][max(kb, xw)] elements: the tile's x rows, one pass or the whole slice (shrink)
//   ys           [RT][ny] elements: the y rows' slices, when staged (expand)
//   then one region used twice:
//     while resolving the tile: scan [2 * SCAN_CAP + 1] ints (segment offsets and slots) and
//                               rank_c / scale_c [RANK_CACHE] (the pool's rank and scale tables)
//     afterwards:               bs [r_alloc][nb] elements, this CTA's B rows when staged
//   Sharing the region keeps a CTA that stages B small enough to sit on an SM beside a CTA of
//   the neighbouring launch.
struct Layout {
  int gbuf, vsm, xs, ys, scan, rank_c, scale_c, bs, ptab, total;
  __host__ __device__ static Layout make(int cs, int rt, int r_alloc, int kb, int nb_staged, int ny, int xw, int npt) {
    Layout L;
    L.gbuf = 128;
    L.vsm = L.gbuf + cs * rt * r_alloc * 4;
    L.xs = (L.vsm + rt * r_alloc * 4 + 127) & ~127;
    L.ys = (L.xs + rt * (xw > kb ? xw : kb) * 2 + 127) & ~127;
    L.scan = (L.ys + rt * ny * 2 + 127) & ~127;
    L.rank_c = L.scan + (2 * SCAN_CAP + 1) * 4;
    L.scale_c = L.rank_c + RANK_CACHE * 4;
    const int resolve_end = L.scale_c + RANK_CACHE * 4;
    L.bs = L.scan;
    const int staged_end = L.bs + r_alloc * nb_staged * 2;
    L.ptab = ((resolve_end > staged_end ? resolve_end : staged_end) + 15) & ~15;
    L.total = L.ptab + npt * 4;
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

// A layout of the same 16 A registers with JN (<= JPW) rank rows per warp: a tile whose rank
// needs fewer rows than the pool's maximum covers 16 / JN chunks of d_in per lane and pass.
template <int JN>
struct Rows {
  static constexpr int value = JN;
};

// Warp reduce-scatter of V partial sums (V a power of two, at most 32): every lane holds V
// partials; afterwards each lane holds the warp's total of value (lane >> (5 - log2 V)), and the
// 32 / V lanes of that group hold the same total. V - 1 + (5 - log2 V) shuffles instead of the
// 5 V of a butterfly per value: at each halving step a lane keeps one half of its values and
// receives its partner's sums of that half.
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&x)[V], int lane) {
#pragma unroll
  for (int cnt = V, s = 16; cnt > 1; cnt >>= 1, s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int k = 0; k < cnt / 2; ++k) {
      const float give = upper ? x[k] : x[k + cnt / 2];
      const float keep = upper ? x[k + cnt / 2] : x[k];
      x[k] = keep + __shfl_xor_sync(0xffffffffu, give, s);
    }
  }
  float t = x[0];
#pragma unroll
  for (int s = 16 / V; s > 0; s >>= 1) t += __shfl_xor_sync(0xffffffffu, t, s);
  return t;
}

template <int DT, int MODE, int RT, int JPW>
__global__ void __launch_bounds__(NTHREADS) decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int UK = Pass<JPW>::UK;
  constexpr int KB = Pass<JPW>::KB;
  const int cs = p.csplit;  // CTAs per tile: the cluster (SHRINK, FUSED) or the N-split (EXPAND)
  const bool stage_b = p.nb > 0;  // B rows of the CTA's slice go to shared memory before the wait
  const Layout L = Layout::make(MODE == MODE_EXPAND ? 1 : cs, RT, p.r_alloc, KB, p.nb, p.ny, p.xw, p.npt);
  uint64_t *xbar = reinterpret_cast<uint64_t *>(smem);
  uint64_t *bbar = xbar + 1;
  uint64_t *ibar = xbar + 2;
  uint64_t *ybar = xbar + 3;
  TileInfo *ti = reinterpret_cast<TileInfo *>(smem + 64);
  float *gbuf = reinterpret_cast<float *>(smem + L.gbuf);
  float *vsm = reinterpret_cast<float *>(smem + L.vsm);
  int32_t *scan = reinterpret_cast<int32_t *>(smem + L.scan);
  int32_t *rank_c = reinterpret_cast<int32_t *>(smem + L.rank_c);
  float *scale_c = reinterpret_cast<float *>(smem + L.scale_c);
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem + L.xs);
  uint16_t *ys = reinterpret_cast<uint16_t *>(smem + L.ys);
  uint16_t *bs = reinterpret_cast<uint16_t *>(smem + L.bs);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool clustered = (MODE != MODE_EXPAND) && cs > 1;
  const uint64_t wlim = p.wait_ns ? p.wait_ns : kWaitLimitNs;  // limit of the waits below
  const uint32_t c = (MODE == MODE_EXPAND) ? (blockIdx.x % cs) : cluster_ctarank();
  const int64_t unit = blockIdx.x / cs;  // (problem, tile)
  const int prob = (int)(unit / p.tiles);
  const int t = (int)(unit % p.tiles);
  const ProblemDev &pr = p.prob[prob];
  const PoolDev &pl = pr.pool;

  // After the tensor-core kernels the launch is sized for the worst case the host can see (every
  // segment just short of tc_min rows): the tiles past the short segments' actual count leave
  // before any setup (tile 0 always stays: it checks the offsets and reports them if malformed).
  if (p.seg_off != nullptr && pr.tc_min > 0 && p.nseg <= SCAN_CAP && t > 0) {
    int32_t *short_tiles = reinterpret_cast<int32_t *>(smem + 120);  // free bytes before gbuf
    if (warp == 0) {
      int32_t n = 0;
      for (int q = lane; q < p.nseg; q += 32) {
        const int32_t len = p.seg_off[q + 1] - p.seg_off[q];
        if (len > 0 && len < pr.tc_min) n += (len + p.rt - 1) / p.rt;
      }
      n = (int32_t)__reduce_add_sync(0xffffffffu, (uint32_t)n);
      if (lane == 0) *short_tiles = n;
    }
    __syncthreads();
    if (t >= *short_tiles) return;  // uniform: the whole block, and every CTA of its cluster
  }

  if (tid == 0) {
    mbar_init(xbar, 1);
    mbar_init(bbar, 1);
    mbar_init(ibar, 1);
    mbar_init(ybar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (clustered) cluster_arrive_relaxed();  // peers may push into our gbuf once everyone arrived
  pdl_launch_dependents();                  // the next kernel may start; it waits for us before reading our outputs

  int32_t *ptab = reinterpret_cast<int32_t *>(smem + L.ptab);
  resolve_tile<MODE>(p, pr, t, ti, scan, rank_c, scale_c, ptab);
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
  // Tiles whose d_in slice fits xs take their x rows (and, when the launcher made room, their
  // y rows) into shared memory by bulk copies issued right after the wait.
  // xs holds XW elements of each row: the CTA's whole d_in slice when the launcher made room
  // (p.xw > 0), else one pass (KB); the whole-slice form is filled by bulk copies.
  const int XW = p.xw > 0 ? p.xw : KB;
  const bool x_bulk = do_shrink && k_end > k_begin && k_end - k_begin <= XW;
  const bool y_bulk = do_expand && p.ny > 0 && n_end > n_begin;
  const uint64_t evict_first = policy_evict_first();
  // Rank rows per warp of this tile's A layout. A one-row tile of the fused kernel whose x slice
  // sits in shared memory and needs several passes of A takes the fewest rows its rank allows (a
  // power of two), so the same registers cover more of d_in per pass -- as long as every pass
  // stays inside the XW elements of xs (guard-free reads). Otherwise the pool's JPW. (The
  // shrink-only kernel keeps JPW: with the smaller layouts it measured slower, 55.6 -> 57.0 us on
  // a 70B q_proj batch with ranks 8..64, and the shrink + expand pair 92.5 -> 97.5 us.)
  int jn = JPW;
  if constexpr (JPW >= 4 && MODE == MODE_FUSED) {
    if (x_bulk && RT == 1 && k_end - k_begin > KB) {
      const int slice = k_end - k_begin;
#pragma unroll
      for (int q = JPW / 2; q >= 1; q >>= 1) {
        const int kbq = 256 * (16 / q);
        if (q * NWARPS >= rank && (slice + kbq - 1) / kbq * kbq <= XW) jn = q;
      }
    }
  }
  const int kbn = 256 * (16 / jn);  // K elements per pass of A in this layout
  // Runs f(Rows<jn>) with jn a compile-time constant (one copy of f per layout in use).
  auto with_rows = [&](auto f) {
    if constexpr (JPW >= 4) {
      if (jn == 1) return f(Rows<1>{});
      if (jn == 2) return f(Rows<2>{});
    }
    if constexpr (JPW >= 8) {
      if (jn == 4) return f(Rows<4>{});
    }
    if constexpr (JPW >= 16) {
      if (jn == 8) return f(Rows<8>{});
    }
    return f(Rows<JPW>{});
  };

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
    }
    if (do_shrink && k_end - k_begin > kbn)
      for (int j = lane; j < rank; j += 32)
        vec_pieces<true>(pl, s, pr.layer, j, k_begin + kbn, k_end, ti->a_tr,
                         [](const uint16_t *src, int, int n) { prefetch_l2(src, (uint32_t)n * 2); });
    if (clustered && lane == 0) mbar_arrive_expect_tx(xbar, (uint32_t)(cs * nr * rank * 4));
  }
  // A registers: in the Rows<JN> layout, register i = jj * (16 / JN) + u holds chunk
  // c8 = lane + 32 u of rank row j = warp + NWARPS jj (a[i / UK][i % UK]; JN = JPW is [jj][u]).
  uint4 a[JPW][UK];
  const bool one_piece_a = pl.kind == MLORA_POOL_STACKED || pl.a_ppv == 1;
  auto load_a = [&](auto rows, int kb0) {
    constexpr int JN = decltype(rows)::value, UKN = 16 / JN;
    const int n8 = min(256 * UKN, k_end - kb0) >> 3;
#pragma unroll
    for (int jj = 0; jj < JN; ++jj) {
      const int j = warp + jj * NWARPS;
      // the vector's start when it lies in one page (stacked pool, square pages): one table read
      // per rank row; else each chunk finds its page
      const uint16_t *base = (j < rank && one_piece_a) ? a_elem(pl, s, pr.layer, j, 0, ti->a_tr) : nullptr;
#pragma unroll
      for (int u = 0; u < UKN; ++u) {
        const int c8 = lane + 32 * u, i = jj * UKN + u;
        const int k = kb0 + c8 * 8;
        // zero outside the slice and the rank: the one-row loop below then needs no guards
        a[i / UK][i % UK] = (j < rank && c8 < n8)
                                ? ldg_stream(one_piece_a ? base + k : a_elem(pl, s, pr.layer, j, k, ti->a_tr), evict_first)
                                : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  if (do_shrink) with_rows([&](auto rows) { load_a(rows, k_begin); });
  if (active && warp == 0 && do_expand && n_end > n_begin) {
      if (b_staged) {
        if (lane == 0) mbar_arrive_expect_tx(bbar, (uint32_t)(rank * (n_end - n_begin) * 2));
        __syncwarp();
        for (int j = lane; j < rank; j += 32)
          vec_pieces<false>(pl, s, pr.layer, j, n_begin, n_end, ti->b_tr, [&](const uint16_t *src, int off, int n) {
            bulk_g2s_hint(bs + j * p.nb + off, src, (uint32_t)n * 2, bbar, evict_first);
          });
      } else if (!(x_bulk && RT == 1 && k_end - k_begin > kbn)) {
        // (a tile that loops over several passes of A prefetches its B rows at its last pass:
        // issued now, they would queue ahead of the later passes' A rows)
        for (int j = lane; j < rank; j += 32)
          vec_pieces<false>(pl, s, pr.layer, j, n_begin, n_end, ti->b_tr,
                            [](const uint16_t *src, int, int n) { prefetch_l2(src, (uint32_t)n * 2); });
      }
  }
  if (x_bulk) {  // the bulk copies fill xs rows < nr up to the slice end; zeros elsewhere (disjoint bytes)
    const int s8 = (k_end - k_begin) >> 3;
    for (int e = tid; e < RT * (XW / 8); e += NTHREADS) {
      const int i = e / (XW / 8), c8 = e % (XW / 8);
      if (i >= nr || c8 >= s8) *reinterpret_cast<uint4 *>(xs + i * XW + c8 * 8) = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  pdl_wait();  // the previous kernel in the stream has finished; its writes are visible
  // The status word is an output: written only after the wait (the previous kernel may be
  // clearing it).
  if (c == 0 && tid == 0 && ti->bad) report(p.status, ti->bad);

  if (tid == 0) {
    if (x_bulk) {
      mbar_arrive_expect_tx(ibar, (uint32_t)(nr * (k_end - k_begin) * 2));
      for (int i = 0; i < nr; ++i)
        bulk_g2s(xs + i * XW, pr.x + (int64_t)(row0 + i) * pr.ldx + k_begin, (uint32_t)(k_end - k_begin) * 2, ibar);
    }
    if (y_bulk) {
      mbar_arrive_expect_tx(ybar, (uint32_t)(nr * (n_end - n_begin) * 2));
      for (int i = 0; i < nr; ++i)
        bulk_g2s(ys + i * p.ny, pr.y + (int64_t)(row0 + i) * pr.ldy + n_begin, (uint32_t)(n_end - n_begin) * 2, ybar);
    }
  }
  int timed_out = 0;

  // ---------------- shrink: partial v over this CTA's slice of d_in ----------------
  if (MODE != MODE_EXPAND) {
    float acc[RT][JPW];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) acc[i][jj] = 0.f;

    if (x_bulk && k_end - k_begin <= KB) {
      // One pass: each lane reads its x chunks from shared memory and meets them with its A
      // chunks in mixed-precision FMAs (16-bit operands, fp32 sums; no unpacking), two chains
      // per (row, rank row). No guards: A is zero outside the slice and the rank, x is zero in
      // rows past nr and past the slice, so every chunk and row runs unconditionally.
      const int ok = mbar_wait(ibar, 0, wlim) ? 1 : 0;
      timed_out = __syncthreads_or(!ok);
      if (!timed_out) {
        float c0[RT][JPW], c1[RT][JPW];
#pragma unroll
        for (int i = 0; i < RT; ++i)
#pragma unroll
          for (int jj = 0; jj < JPW; ++jj) c0[i][jj] = c1[i][jj] = 0.f;
#pragma unroll
        for (int u = 0; u < UK; ++u) {
#pragma unroll
          for (int i = 0; i < RT; ++i) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xs + i * XW + (lane + 32 * u) * 8);
#pragma unroll
            for (int jj = 0; jj < JPW; ++jj) mfma8<DT>(xv, a[jj][u], c0[i][jj], c1[i][jj]);
          }
        }
#pragma unroll
        for (int i = 0; i < RT; ++i)
#pragma unroll
          for (int jj = 0; jj < JPW; ++jj) acc[i][jj] = c0[i][jj] + c1[i][jj];
      }
    } else if (x_bulk && RT == 1) {
      // The x slice is in shared memory; A comes in passes of KB elements (the first loaded into
      // registers before the wait, the next ones from L2, where they were prefetched). No
      // guards: A is zero outside the slice and the rank, x is zero past the slice and nr.
      const int ok = mbar_wait(ibar, 0, wlim) ? 1 : 0;
      timed_out = __syncthreads_or(!ok);
      float c0[JPW], c1[JPW];  // two chains per rank row, across the passes
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) c0[jj] = c1[jj] = 0.f;
      with_rows([&](auto rows) {
        constexpr int JN = decltype(rows)::value, UKN = 16 / JN, KBN = 256 * UKN;
        for (int pass = 0; !timed_out && pass * KBN < k_end - k_begin; ++pass) {
          if (pass > 0) load_a(rows, k_begin + pass * KBN);
          const uint16_t *xp = xs + pass * KBN;  // pass < ceil(slice / KBN), so xp + KBN <= xs + XW
          // B rows of a tile with several passes are prefetched at its last one (a one-pass tile
          // prefetched them before the wait)
          if (pass > 0 && !b_staged && do_expand && n_end > n_begin && (pass + 1) * KBN >= k_end - k_begin)
            for (int j = tid; j < rank; j += NTHREADS)
              vec_pieces<false>(pl, s, pr.layer, j, n_begin, n_end, ti->b_tr,
                                [](const uint16_t *src, int, int n) { prefetch_l2(src, (uint32_t)n * 2); });
#pragma unroll
          for (int u = 0; u < UKN; ++u) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xp + (lane + 32 * u) * 8);
#pragma unroll
            for (int jj = 0; jj < JN; ++jj) {
              const int i = jj * UKN + u;
              mfma8<DT>(xv, a[i / UK][i % UK], c0[jj], c1[jj]);
            }
          }
        }
      });
      // rank rows jj >= JN of this layout lie past the rank: their sums stay zero
#pragma unroll
      for (int jj = 0; jj < JPW; ++jj) acc[0][jj] = c0[jj] + c1[jj];
    } else if (do_shrink) {
      for (int kb0 = k_begin; kb0 < k_end; kb0 += KB) {
        const int n8 = min(KB, k_end - kb0) >> 3;
        if (kb0 != k_begin) load_a(Rows<JPW>{}, kb0);
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

    // Warp-level sums of the RT x JPW dot products (value q = i * JPW + jj): after the
    // reduce-scatter, lane l holds the total of value l / LPV, in LPV replicas (lanes with the
    // same value); V = RT * JPW partials, taken 32 at a time.
    constexpr int V = RT * JPW;
    constexpr int VG = V < 32 ? V : 32;  // values per reduce-scatter
    constexpr int NG = V / VG;           // groups of 32 values (RT 4 x JPW 16: 2)
    constexpr int LPV = 32 / VG;         // lanes per value
    float tot[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float part[VG];
#pragma unroll
      for (int k = 0; k < VG; ++k) part[k] = acc[(g * VG + k) / JPW][(g * VG + k) % JPW];
      tot[g] = warp_reduce_scatter<VG>(part, lane);
    }
    const int myq = lane / LPV, rep = lane % LPV;  // this lane's value (within a group) and replica

    if (clustered) {
      // Push this CTA's partials into slot c of every peer's gather buffer: replica r of a value
      // pushes it to peers r, r + LPV, ... A CTA that timed out pushes nothing; its peers then
      // time out too and skip the tile.
      cluster_wait();  // every peer has initialised its exchange barrier
      if (do_shrink && !timed_out) {
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const int q = g * VG + myq, i = q / JPW, jj = q % JPW;
          const int j = warp + jj * NWARPS;
          if (j < rank && i < nr) {
            for (int peer = rep; peer < cs; peer += LPV)
              st_async_f32(dsmem_addr(gbuf + (c * RT + i) * p.r_alloc + j, peer), tot[g], dsmem_addr(xbar, peer));
          }
        }
      }
      if (do_shrink) {
        const int ok = mbar_wait_cluster(xbar, 0, wlim) ? 1 : 0;
        timed_out |= __syncthreads_or(!ok);
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
      // Every push into this CTA has landed (or the wait gave up, and the exit drains it): the
      // CTA needs nothing more from its peers and its shared memory is no longer written by them.
    } else if (do_shrink && !timed_out && rep == 0) {
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const int q = g * VG + myq, i = q / JPW, jj = q % JPW;
        const int j = warp + jj * NWARPS;
        if (j < rank && i < nr) {
          if (MODE == MODE_SHRINK) pr.v[(int64_t)(row0 + i) * pl.r_max + j] = tot[g];
          else vsm[i * p.r_alloc + j] = tot[g];
        }
      }
    }
  } else if (active) {
    // expand only: this tile's v rows from global memory (written by the previous kernel)
    for (int e = tid; e < nr * rank; e += NTHREADS) {
      const int i = e / rank, j = e % rank;
      vsm[i * p.r_alloc + j] = pr.v[(int64_t)(row0 + i) * pl.r_max + j];
    }
  }
  // v is published to every thread by this barrier, which also agrees on the staged B rows and
  // the staged y slice having landed.
  {
    int ok = 1;
    if (b_staged && !timed_out) ok &= mbar_wait(bbar, 0, wlim) ? 1 : 0;
    if (y_bulk && !timed_out) ok &= mbar_wait(ybar, 0, wlim) ? 1 : 0;
    timed_out |= __syncthreads_or(!ok);
  }

  // ---------------- expand: y[rows][this CTA's slice of d_out] ----------------
  if (do_expand && !timed_out) {
    const int n8 = (n_end - n_begin) >> 3;
    if (RT == 1) {
      // One row: 8 columns per thread and pass, rank rows summed with the paired fp32 FMA in
      // two chains (even and odd rank rows); v sits in registers for ranks up to 16.
      constexpr bool VREG = JPW <= 2;
      constexpr int RV = VREG ? 8 * JPW : 1;
      float vr[RV];
#pragma unroll
      for (int j = 0; j < RV; ++j) vr[j] = (VREG && j < rank) ? vsm[j] : 0.f;
      for (int c8 = tid; c8 < n8; c8 += NTHREADS) {
        const int n0 = n_begin + c8 * 8;
        const BRows brow(pl, s, pr.layer, n0, ti->b_tr);
        float2 ev[4], od[4];  // even / odd rank rows
#pragma unroll
        for (int e = 0; e < 4; ++e) ev[e] = od[e] = make_float2(0.f, 0.f);
        auto add_row = [&](const uint4 &bw, float vj, float2 (&acc2)[4]) {
          float2 b2[4];
          unpack8x2<DT>(bw, b2);
          const float2 v2 = make_float2(vj, vj);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[e] = __ffma2_rn(v2, b2[e], acc2[e]);
        };
        // B rows in flight per thread when they come from global memory: 16 above rank 16 (half
        // the round trips to L2; the A registers are free by now)
        constexpr int UB = VREG ? 8 : 16;
        if constexpr (VREG) {
          if (b_staged && rank == RV) {  // every rank row present: straight-line, no guards
#pragma unroll
            for (int j = 0; j < RV; j += 2) {
              add_row(*reinterpret_cast<const uint4 *>(bs + j * p.nb + c8 * 8), vr[j], ev);
              add_row(*reinterpret_cast<const uint4 *>(bs + (j + 1) * p.nb + c8 * 8), vr[j + 1], od);
            }
          } else if (b_staged) {
#pragma unroll
            for (int j = 0; j < RV; j += 2) {
              if (j < rank) add_row(*reinterpret_cast<const uint4 *>(bs + j * p.nb + c8 * 8), vr[j], ev);
              if (j + 1 < rank) add_row(*reinterpret_cast<const uint4 *>(bs + (j + 1) * p.nb + c8 * 8), vr[j + 1], od);
            }
          } else {
#pragma unroll
            for (int j0 = 0; j0 < RV; j0 += UB) {
              uint4 bq[UB];
              if (j0 + UB <= rank) {  // a whole batch of rank rows: no guards
#pragma unroll
                for (int u = 0; u < UB; ++u) bq[u] = ldg_stream(brow(j0 + u), evict_first);
#pragma unroll
                for (int u = 0; u < UB; u += 2) {
                  add_row(bq[u], vr[j0 + u], ev);
                  add_row(bq[u + 1], vr[j0 + u + 1], od);
                }
              } else if (j0 < rank) {
#pragma unroll
                for (int u = 0; u < UB; ++u)
                  if (j0 + u < rank) bq[u] = ldg_stream(brow(j0 + u), evict_first);
#pragma unroll
                for (int u = 0; u < UB; u += 2) {
                  if (j0 + u < rank) add_row(bq[u], vr[j0 + u], ev);
                  if (j0 + u + 1 < rank) add_row(bq[u + 1], vr[j0 + u + 1], od);
                }
              }
            }
          }
        } else {
          if (b_staged) {
#pragma unroll 2
            for (int j = 0; j < rank; j += 2) {
              add_row(*reinterpret_cast<const uint4 *>(bs + j * p.nb + c8 * 8), vsm[j], ev);
              if (j + 1 < rank) add_row(*reinterpret_cast<const uint4 *>(bs + (j + 1) * p.nb + c8 * 8), vsm[j + 1], od);
            }
          } else {
            for (int j0 = 0; j0 < rank; j0 += UB) {
              uint4 bq[UB];
              if (j0 + UB <= rank) {  // a whole batch of rank rows: no guards
#pragma unroll
                for (int u = 0; u < UB; ++u) bq[u] = ldg_stream(brow(j0 + u), evict_first);
#pragma unroll
                for (int u = 0; u < UB; u += 2) {
                  add_row(bq[u], vsm[j0 + u], ev);
                  add_row(bq[u + 1], vsm[j0 + u + 1], od);
                }
              } else {
#pragma unroll
                for (int u = 0; u < UB; ++u)
                  if (j0 + u < rank) bq[u] = ldg_stream(brow(j0 + u), evict_first);
#pragma unroll
                for (int u = 0; u < UB; u += 2) {
                  if (j0 + u < rank) add_row(bq[u], vsm[j0 + u], ev);
                  if (j0 + u + 1 < rank) add_row(bq[u + 1], vsm[j0 + u + 1], od);
                }
              }
            }
          }
        }
        const uint4 yw = y_bulk ? *reinterpret_cast<const uint4 *>(ys + c8 * 8) : ldg_u4(pr.y + (int64_t)row0 * pr.ldy + n0);
        float yf[8];
        unpack8<DT>(yw, yf);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          yf[2 * e] = fmaf(scale, ev[e].x + od[e].x, yf[2 * e]);
          yf[2 * e + 1] = fmaf(scale, ev[e].y + od[e].y, yf[2 * e + 1]);
        }
        *reinterpret_cast<uint4 *>(pr.y + (int64_t)row0 * pr.ldy + n0) = pack8<DT>(yf);
      }
    } else {
      // Several rows: per rank row, the B chunk is unpacked once and meets every row's v (a
      // broadcast read of shared memory) in paired fp32 FMAs.
      for (int c8 = tid; c8 < n8; c8 += NTHREADS) {
        const int n0 = n_begin + c8 * 8;
        const BRows brow(pl, s, pr.layer, n0, ti->b_tr);
        float2 acc2[RT][4];
#pragma unroll
        for (int i = 0; i < RT; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[i][e] = make_float2(0.f, 0.f);
        auto add_row = [&](const uint4 &bw, int j) {
          float2 b2[4];
          unpack8x2<DT>(bw, b2);
#pragma unroll
          for (int i = 0; i < RT; ++i) {
            const float vij = vsm[i * p.r_alloc + j];  // rows past nr hold garbage; never stored
            const float2 v2 = make_float2(vij, vij);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc2[i][e] = __ffma2_rn(v2, b2[e], acc2[i][e]);
          }
        };
        constexpr int RF = 8 * JPW;  // largest rank of this instantiation
        if (b_staged && rank == RF && RF <= 16) {  // every rank row present: straight-line, no guards
#pragma unroll
          for (int j = 0; j < RF; ++j) add_row(*reinterpret_cast<const uint4 *>(bs + j * p.nb + c8 * 8), j);
        } else if (b_staged) {
#pragma unroll 2
          for (int j = 0; j < rank; ++j) add_row(*reinterpret_cast<const uint4 *>(bs + j * p.nb + c8 * 8), j);
        } else {
          constexpr int UB = 4;  // B loads in flight per thread
          for (int j0 = 0; j0 < rank; j0 += UB) {
            uint4 b[UB];
#pragma unroll
            for (int u = 0; u < UB; ++u)
              if (j0 + u < rank) b[u] = ldg_stream(brow(j0 + u), evict_first);
#pragma unroll
            for (int u = 0; u < UB; ++u)
              if (j0 + u < rank) add_row(b[u], j0 + u);
          }
        }
#pragma unroll
        for (int i = 0; i < RT; ++i) {
          if (i < nr) {
            float yf[8];
            unpack8<DT>(y_bulk ? *reinterpret_cast<const uint4 *>(ys + i * p.ny + c8 * 8)
                               : ldg_u4(pr.y + (int64_t)(row0 + i) * pr.ldy + n0), yf);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              yf[2 * e] = fmaf(scale, acc2[i][e].x, yf[2 * e]);
              yf[2 * e + 1] = fmaf(scale, acc2[i][e].y, yf[2 * e + 1]);
            }
            *reinterpret_cast<uint4 *>(pr.y + (int64_t)(row0 + i) * pr.ldy + n0) = pack8<DT>(yf);
          }
        }
      }
    }
  }

  // Copies still in flight after a time-out land before the CTA exits (bounded waits), and so do
  // the peers' pushes into this CTA's exchange buffer (a peer that gave up before pushing never
  // completes that barrier: the wait then ends at its limit).
  if (timed_out) {
    if (b_staged) (void)mbar_wait(bbar, 0, kDrainLimitNs);
    if (x_bulk) (void)mbar_wait(ibar, 0, kDrainLimitNs);
    if (y_bulk) (void)mbar_wait(ybar, 0, kDrainLimitNs);
    if (clustered && do_shrink) (void)mbar_wait_cluster(xbar, 0, kDrainLimitNs);
    if (tid == 0) report(p.status, MLORA_STATUS_TIMEOUT);
  }
}

// Host: launch one instantiation with the cluster and PDL attributes.
template <int DT, int MODE, int RT, int JPW>
cudaError_t launch_one(const DecodeParams &p, unsigned grid, size_t smem, int cluster, bool pdl, cudaStream_t stream) {
  auto kern = decode_kernel<DT, MODE, RT, JPW>;
  // Kernel attributes are per device: the dynamic shared memory this instantiation was set up
  // for on each device. An entry is raised only after the attribute calls behind it returned,
  // so a thread that reads it large enough may launch at once.
  static std::atomic<int> configured_smem[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  if (dev >= kMaxDevices || configured_smem[dev].load(std::memory_order_acquire) < (int)smem) {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= kMaxDevices || configured_smem[dev].load(std::memory_order_relaxed) < (int)smem) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      if (dev < kMaxDevices) configured_smem[dev].store((int)smem, std::memory_order_release);
    }
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
  if (r <= 16) return launch_one<DT, MODE, 4, 2>(p, grid, smem, cluster, pdl, stream);
  if (r <= 32) return launch_one<DT, MODE, 4, 4>(p, grid, smem, cluster, pdl, stream);
  if (r <= 64) return launch_one<DT, MODE, 4, 8>(p, grid, smem, cluster, pdl, stream);
  return launch_one<DT, MODE, 4, 16>(p, grid, smem, cluster, pdl, stream);
}

}  // namespace decode
}  // namespace mlora
