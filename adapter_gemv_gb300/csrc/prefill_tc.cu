// prefill_tc.cu -- tensor-core path for long SGMV segments (prefill), sm_103a.
//
// A long segment that shares one adapter is a real dense contraction: many rows against one
// adapter's narrow matrices, a GEMM rather than a batch of GEMVs ("Multi-LoRA Serving, in depth",
// section "Two shapes: SGMV for prefill, BGMV for decode"; Punica section 3.4, "Tensor Core
// usage"). Segments of at least tc_min rows (the host's choice per call, 8 to 32) run here in
// tiles of at most 128 rows, the last one masked; shorter segments run on the CUDA-core kernels. bf16 and fp16 stacked pools; the MMAs are kind::f16 with both operands of
// the pool's type and fp32 accumulators.
//
//   shrink  V[128 x r] = X[128 x d_in] . A   : one CTA per (tile, K part); a cluster of K parts
//           sums its fp32 partials through distributed shared memory. X tiles and A^T rows are
//           both K-major; TMA (128-byte swizzle) feeds an mbarrier ring as deep as shared memory
//           allows, two swizzle atoms (128 K elements) per stage; one thread issues tcgen05.mma
//           (M = 128, N = rank rounded up to 16, K = 16 per instruction) into a TMEM accumulator,
//           and all four warps read it back with tcgen05.ld.
//   expand  Y[128 x 64] += scale . V[128 x r] . B[r x 64] per block : one CTA per (tile, run of
//           64-column blocks), in warp roles: a producer lane TMA-loads each block's y tile and B
//           rows into a ring of buffers, an MMA lane multiplies into one of two TMEM accumulators,
//           eight epilogue warps add the result into the y tile in shared memory (rounded once),
//           and a store lane TMA-stores it and frees the buffer. V (fp32) is split into hi + lo
//           parts of the pool's type, both multiplied into the fp32 accumulator; fp16 rows of V are
//           first scaled by a power of two so that they cannot overflow.
// Every wait is bounded; a timed-out CTA reports MLORA_STATUS_TIMEOUT and writes nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace mlora {

namespace {

constexpr int BM = 128;      // MMA M; a tile holds p.bm <= BM rows (the host's chunk size)
constexpr int kMinTileRows = 64;  // smallest chunk the host picks
constexpr int BK = 64;       // K elements per stage (one 128-byte swizzle row)
constexpr int SKA = 2;  // shrink: swizzle atoms (64 K elements each) per ring stage: 256 contiguous
                        // bytes of each x row per stage (measured 2.5 % faster than one atom)
constexpr int MAX_STAGES = 12;  // shrink ring depth: as many stages as fit, up to this
constexpr int MAX_EBUF = 8;  // expand pipeline buffers: as many as fit with two CTAs per SM, up to this
constexpr int NTHREADS = 128;
constexpr int SCAN_CAP = 512;
constexpr int kTcBatchRows = 256;  // rows in a batch below which the tensor cores are not tried
constexpr int kTcAvgRows = 8;      // average rows per segment below which they are not tried

struct TcTile {
  int32_t row0, nr, slot, rank, skip, bad;
  float scale;
};

// Tile t = the t-th block of p.bm rows, walking the segments in order: a segment of at least
// p.tc_min rows contributes ceil(len / bm) blocks (the last one may be partial: nr < bm);
// shorter segments belong to the CUDA-core kernels. Whole block participates; row metadata only.
// A pool of at most blockDim.x slots has its rank and scale tables loaded at the start, beside the
// offsets (one round trip to memory instead of two).
__device__ void resolve_tc_tile(const TcParams &p, int t, TcTile *ti, int32_t *scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool cached = p.num_slots <= (int)blockDim.x;
  int32_t my_rank = 0;
  float my_scale = 0.f;
  if (cached && tid < p.num_slots) {
    my_rank = p.rank[tid];
    my_scale = p.scale[tid];
  }
  if (tid == 0) {
    ti->skip = 1;
    ti->bad = 0;
    ti->slot = -2;
  }
  __syncthreads();
  int32_t carry = 0, found = 0, bad = 0;
  for (int base = 0; base < p.nseg; base += SCAN_CAP) {
    const int cnt = min(SCAN_CAP, p.nseg - base);
    for (int q = tid; q <= cnt; q += (int)blockDim.x) {
      scan[q] = p.seg_off[base + q];
      if (q < cnt) scan[SCAN_CAP + 1 + q] = p.seg_slot[base + q];
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
        }
        const int32_t nt = (q < cnt && len >= p.tc_min && len > 0) ? (len + p.bm - 1) / p.bm : 0;
        int32_t incl = nt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += o;
        }
        const int32_t excl = carry + incl - nt;
        const bool mine = q < cnt && t >= excl && t < excl + nt;
        if (!found && mine) {
          ti->row0 = lo + (t - excl) * p.bm;
          ti->nr = min(p.bm, len - (t - excl) * p.bm);
          ti->slot = scan[SCAN_CAP + 1 + q];
        }
        found |= __any_sync(0xffffffffu, mine);
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      bad = __any_sync(0xffffffffu, bad);
    }
    __syncthreads();
  }
  if (cached) {  // the thread of the tile's slot hands over the rank and scale it loaded
    const int s = ti->slot;
    if (s >= 0 && s == tid) {
      ti->rank = my_rank;
      ti->scale = my_scale;
    }
    __syncthreads();
  }
  if (tid == 0) {
    int32_t b = bad ? MLORA_STATUS_BAD_OFFSETS : 0;
    int skip = (!found || b) ? 1 : 0;
    if (!skip) {
      const int s = ti->slot;
      if (s == -1) {
        skip = 1;
      } else if (s < -1 || s >= p.num_slots) {
        b = MLORA_STATUS_BAD_SLOT;
        skip = 1;
      } else {
        const int r = cached ? ti->rank : p.rank[s];
        if (r < 1 || r > p.r_max) {
          b = MLORA_STATUS_BAD_RANK;
          skip = 1;
        } else {
          ti->rank = r;
          ti->scale = cached ? ti->scale : p.scale[s];
        }
      }
    }
    ti->bad = b;
    ti->skip = skip;
  }
  __syncthreads();
}

// Paged pools: the page ids of the tile's vectors (rows j < rpad of A^T or of B, for the tile's slot
// and layer), ptab[j * ppv + q] = page of the q-th piece of vector j, -1 for j >= rank (those rows
// are zero-filled). Whole block; true if a page id lies outside the pool (BAD_PAGE).
__device__ bool load_page_ids(const TcParams &p, const int32_t *tab, int ppv, int s, int rank, int32_t *ptab) {
  const int64_t t0 = ((int64_t)s * p.num_layers + p.layer) * p.r_max;
  int bad = 0;
  for (int e = threadIdx.x; e < p.rpad * ppv; e += blockDim.x) {
    int32_t pg = -1;
    if (e / ppv < rank) {
      pg = tab[t0 * ppv + e];
      bad |= (pg < 0 || pg >= p.num_pages) ? 1 : 0;
    }
    ptab[e] = pg;
  }
  return __syncthreads_or(bad) != 0;
}

// Paged pools: one 64-element K-major (A^T) or MN-major (B) atom of rows j < rpad, elements
// [e0, e0 + 64) of each vector (d elements long), copied by the calling warp with 16-byte cp.async
// into the 128-byte-swizzled layout a TMA load would write (row j at j * 128, chunk cc at
// (cc ^ (j % 8)) * 16). Chunks past the vector's end or of rows j >= rank are zero-filled. A
// piece of 8 elements never straddles pages (page_elems is a multiple of 8, at least 64, so an
// atom crosses at most one page boundary).
__device__ __forceinline__ void gather_atom(const TcParams &p, const int32_t *ptab, int ppv, int d, int e0,
                                            uint8_t *dst, int lane) {
  const int pe = p.page_elems;
  const int pq = e0 / pe, rq = e0 - pq * pe;
  for (int e = lane; e < p.rpad * 8; e += 32) {
    const int j = e >> 3, cc = e & 7;
    int off = rq + cc * 8, pidx = pq;
    if (off >= pe) {
      off -= pe;
      ++pidx;
    }
    const int32_t pg = (e0 + cc * 8 < d) ? ptab[j * ppv + pidx] : -1;
    const uint16_t *src = pg >= 0 ? p.pages + (int64_t)pg * pe + off : p.pages;
    tc::cp_async16(dst + j * 128 + ((cc ^ (j & 7)) << 4), src, pg >= 0 ? 16u : 0u);
  }
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------------------------------
// shrink

struct ShrinkSmem {
  int stages, stage_bytes, a_off, bar_off, total;
  // A stage holds the SKA swizzle atoms of the X tile (bm rows of 128 B each, atom q at
  // q * bm * 128) and then those of the A^T rows (rpad rows each). The MMA reads 128 rows from
  // an X atom: for bm < 128 the rows past bm are whatever follows in shared memory (their sums
  // land in accumulator rows that are never stored); the pad after the ring keeps every such
  // read inside the allocation.
  // stages = 0: as many as fit in 227 KB (a deep ring keeps one CTA's TMA loads streaming)
  __host__ __device__ static ShrinkSmem make(int rpad, int bm, int stages = 0) {
    ShrinkSmem L;
    L.a_off = SKA * bm * BK * 2;
    L.stage_bytes = (L.a_off + SKA * rpad * BK * 2 + 1023) & ~1023;
    const int overhang = (SKA - 1) * bm * 128 + BM * 128 - L.stage_bytes;  // last atom's 128-row read
    const int pad = overhang > 0 ? (overhang + 1023) & ~1023 : 0;
    const int fixed = 1024 + (2 * SCAN_CAP + 1) * 4 + 1024;  // barriers, tile info, scan, alignment slack
    if (stages <= 0) stages = (227 * 1024 - fixed - pad) / L.stage_bytes;
    L.stages = stages < 2 ? 2 : stages > MAX_STAGES ? MAX_STAGES : stages;
    L.bar_off = L.stages * L.stage_bytes + pad;
    L.total = L.bar_off + fixed;
    return L;
  }
};

template <int DT>
__global__ void __launch_bounds__(NTHREADS) tc_shrink_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                             const __grid_constant__ CUtensorMap tm_a,
                                                             const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const ShrinkSmem L = ShrinkSmem::make(p.rpad, p.bm, p.stages);
  const int STAGES = L.stages;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  uint64_t *empty = full + MAX_STAGES;
  uint64_t *accbar = empty + MAX_STAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accbar + 1);
  int32_t *flags = reinterpret_cast<int32_t *>(tmem_slot + 1);  // [0] = timed out
  TcTile *ti = reinterpret_cast<TcTile *>(smem + L.bar_off + 256);
  int32_t *scan = reinterpret_cast<int32_t *>(smem + L.bar_off + 1024);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ks = p.ksplit;
  const uint32_t c = cluster_ctarank();
  const int t = blockIdx.y;
  const uint32_t ncols = p.tmem_cols;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], p.paged ? 1 + 32 : 1);  // paged: + one cp.async arrival per producer lane
      mbar_init(&empty[s], 1);
    }
    mbar_init(accbar, 1);
    flags[0] = 0;
    mbar_fence_init();
    tc::tma_prefetch_desc(&tm_x);
    tc::tma_prefetch_desc(&tm_a);
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, ncols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the expand of a fused call may start now: it reads v only after waiting for this grid
  pdl_launch_dependents();

  resolve_tc_tile(p, t, ti, scan);
  int32_t *ptab = scan;  // paged: the scan area is free after the resolve
  bool active = !ti->skip;
  int32_t bad = ti->bad;
  if (p.paged && active && load_page_ids(p, p.a_tab, p.a_ppv, ti->slot, ti->rank, ptab)) {
    bad |= MLORA_STATUS_BAD_PAGE;
    active = false;
  }
  if (c == 0 && tid == 0 && bad) report(p.status, bad);
  const int row0 = ti->row0, nr = ti->nr, s = ti->slot, rank = ti->rank;
  const int kb_total = (p.d_in + SKA * BK - 1) / (SKA * BK);
  const int kb_per = (kb_total + ks - 1) / ks;
  const int kb0 = min((int)c * kb_per, kb_total), kb1 = min(kb0 + kb_per, kb_total);
  const int nkb = active ? kb1 - kb0 : 0;
  const int arow = (s * p.num_layers + p.layer) * p.r_max;
  // bytes the stage's TMA loads bring: the X tile, and the A^T rows unless they are gathered
  const uint32_t stage_tx = (uint32_t)(SKA * (p.bm * BK * 2 + (p.paged ? 0 : p.rpad * BK * 2)));
  const uint32_t idesc = tc::idesc_f16(DT == MLORA_BF16, false, false, BM, p.rpad);

  if (warp == 0 && p.paged) {
    // producer (whole warp): lane 0 TMA-loads the X tile of each K block, and the warp gathers the
    // A^T rows from their pages with cp.async (completing on the same barrier)
    for (int i = 0; i < nkb; ++i) {
      const int st = i % STAGES;
      const int ok = (i < STAGES || mbar_wait(&empty[st], (uint32_t)((i / STAGES) - 1) & 1u)) ? 1 : 0;
      if (__any_sync(0xffffffffu, !ok)) {
        if (lane == 0) flags[0] = 1;
        break;
      }
      uint8_t *sb = smem + st * L.stage_bytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[st], stage_tx);
        for (int q = 0; q < SKA; ++q)
          tc::tma_load_2d(sb + q * p.bm * 128, &tm_x, ((kb0 + i) * SKA + q) * BK, row0, &full[st]);
      }
      for (int q = 0; q < SKA; ++q)
        gather_atom(p, ptab, p.a_ppv, p.d_in, ((kb0 + i) * SKA + q) * BK, sb + L.a_off + q * p.rpad * 128, lane);
      tc::cp_async_arrive(&full[st]);
    }
    // nothing may land in shared memory after the CTA exits: the last stages' copies (bounded)
    if (lane == 0)
      for (int i = max(nkb - STAGES, 0); i < nkb; ++i)
        (void)mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u, kDrainLimitNs);
    __syncwarp();
  } else if (warp == 0) {
    // producer (one lane): TMA X tile and A^T rows of each K block into the ring
    for (int i = 0; lane == 0 && i < nkb; ++i) {
      const int st = i % STAGES;
      if (i >= STAGES && !mbar_wait(&empty[st], (uint32_t)((i / STAGES) - 1) & 1u)) {
        flags[0] = 1;
        break;
      }
      uint8_t *sb = smem + st * L.stage_bytes;
      mbar_arrive_expect_tx(&full[st], stage_tx);
      for (int q = 0; q < SKA; ++q) {
        tc::tma_load_2d(sb + q * p.bm * 128, &tm_x, ((kb0 + i) * SKA + q) * BK, row0, &full[st]);
        tc::tma_load_2d(sb + L.a_off + q * p.rpad * 128, &tm_a, ((kb0 + i) * SKA + q) * BK, arow, &full[st]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer (one lane)
    for (int i = 0; lane == 0 && i < nkb; ++i) {
      const int st = i % STAGES;
      if (!mbar_wait(&full[st], (uint32_t)(i / STAGES) & 1u)) {
        flags[0] = 1;
        break;
      }
      if (p.paged) tc::fence_proxy_async();  // the cp.async-gathered A^T rows -> the tensor cores
      tc::tc_fence_after();
      const uint8_t *sb = smem + st * L.stage_bytes;
#pragma unroll
      for (int k = 0; k < SKA * BK / 16; ++k) {
        const int q = k / (BK / 16), kk = k % (BK / 16);
        const uint64_t da = tc::smem_desc_sw128(sb + q * p.bm * 128 + kk * 32, 16, 1024);
        const uint64_t db = tc::smem_desc_sw128(sb + L.a_off + q * p.rpad * 128 + kk * 32, 16, 1024);
        tc::mma_f16(tmem, da, db, idesc, (i > 0 || k > 0) ? 1u : 0u);
      }
      tc::mma_commit(&empty[st]);
    }
    if (lane == 0 && nkb > 0) tc::mma_commit(accbar);
    __syncwarp();
  }
  __syncthreads();

  // epilogue: TMEM row m (lane) of this warp's quarter -> v (or the cluster reduction buffer)
  int ok = 1;
  if (nkb > 0) ok = mbar_wait(accbar, 0) ? 1 : 0;
  const int timed_out = __syncthreads_or(!ok || flags[0]);
  tc::tc_fence_after();
  // The ring is idle now. It holds the tile's v rows: [128][rpad] fp32 partials for the cluster
  // sum, or (no K split) [128][rpad + 4] for the copy out, which writes whole rows of v with
  // 16-byte stores (thread m writing its own row would scatter 4-byte stores over 128 rows).
  float *red = reinterpret_cast<float *>(smem);
  const int m = warp * 32 + lane;
  const int rs_ = ks == 1 ? p.rpad + 4 : p.rpad;  // row stride in red (floats)
  if (active && !timed_out) {
    for (int c16 = 0; c16 < p.rpad / 16; ++c16) {
      float vals[16];
      if (nkb > 0) {
        tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c16 * 16), vals);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) vals[e] = 0.f;
      }
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4)
        *reinterpret_cast<float4 *>(red + m * rs_ + c16 * 16 + e4 * 4) =
            make_float4(vals[e4 * 4], vals[e4 * 4 + 1], vals[e4 * 4 + 2], vals[e4 * 4 + 3]);
    }
    if (ks == 1) {
      __syncthreads();  // uniform: active and timed_out are the block's
      const bool vec = (p.r_max & 3) == 0 && (reinterpret_cast<uintptr_t>(p.v) & 15) == 0;
      if (vec) {
        const int rq = (rank + 3) >> 2;  // 4-float groups per row
        for (int e = tid; e < nr * rq; e += NTHREADS) {
          const int row = e / rq, j = (e - row * rq) * 4;
          float *dst = p.v + (int64_t)(row0 + row) * p.r_max + j;
          const float4 val = *reinterpret_cast<const float4 *>(red + row * rs_ + j);
          if (j + 4 <= rank) {
            *reinterpret_cast<float4 *>(dst) = val;
          } else {
            dst[0] = val.x;
            if (j + 1 < rank) dst[1] = val.y;
            if (j + 2 < rank) dst[2] = val.z;
          }
        }
      } else {
        for (int e = tid; e < nr * rank; e += NTHREADS) {
          const int row = e / rank, j = e - row * rank;
          p.v[(int64_t)(row0 + row) * p.r_max + j] = red[row * rs_ + j];
        }
      }
    }
  }
  if (ks > 1) {
    cluster_sync();
    if (active && !timed_out) {
      // CTA c sums rows [c * rp, min(128, (c + 1) * rp)) over the cluster, in rank order
      const int rp = (p.bm + ks - 1) / ks;
      const int m_lo = min((int)c * rp, nr), m_hi = min(m_lo + rp, nr);
      for (int e = tid; e < (m_hi - m_lo) * rank; e += NTHREADS) {
        const int mm = m_lo + e / rank, j = e % rank;
        float sum = 0.f;
        for (int q = 0; q < ks; ++q) sum += dsmem_ld_f32(dsmem_addr(&red[mm * p.rpad + j], q));
        p.v[(int64_t)(row0 + mm) * p.r_max + j] = sum;
      }
    }
    cluster_sync();
  }
  if (timed_out && tid == 0) report(p.status, MLORA_STATUS_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, ncols);
}

// ------------------------------------------------------------------------------------------
// expand

// Warp roles: warps 0-7 run the epilogue -- warp w reads TMEM lanes 32 (w % 4) .. +31 (its 32 y
// rows) and the block's columns 32 (w / 4) .. +31; warps 0-3 also build V, one row per thread;
// warp 8 lane 0 loads (TMA) the y tile and B rows of each 64-column block into a ring of
// buffers; warp 9 lane 0 issues the MMAs into one of two TMEM accumulators, so a block's MMA
// overlaps the previous block's epilogue; warp 10 lane 0 stores each finished y tile (TMA) and
// frees its buffer once the store has read it, so the epilogue goes on to the next block at once.
constexpr int EXP_EPI_WARPS = 8;
constexpr int EXP_THREADS = (EXP_EPI_WARPS + 3) * 32;

// Shared memory: EBUF pipeline buffers, each with the y tile of one 64-column block (bm rows x
// 128 B) followed by its B rows (one MN atom: rpad K rows x 128 B). V (the MMA's A operand) lives in
// tensor memory, which leaves the shared memory to the ring.
struct ExpandSmem {
  int nbuf, buf_off, buf_bytes, b_in_buf, bar_off, total;
  // nbuf = 0: as many buffers as fit in `budget` bytes
  __host__ __device__ static ExpandSmem make(int rpad, int bm, int nbuf = 0, int budget = 227 * 1024) {
    ExpandSmem L;
    L.buf_off = 0;
    L.b_in_buf = bm * 128;
    L.buf_bytes = (L.b_in_buf + rpad * 128 + 1023) & ~1023;
    const int fixed = 1024 + (2 * SCAN_CAP + 1) * 4 + 1024;
    if (nbuf <= 0) nbuf = (budget - fixed - L.buf_off) / L.buf_bytes;
    L.nbuf = nbuf < 2 ? 2 : nbuf > MAX_EBUF ? MAX_EBUF : nbuf;
    L.bar_off = L.buf_off + L.nbuf * L.buf_bytes;
    L.total = L.bar_off + fixed;
    return L;
  }
};

constexpr int EBN = 64;  // expand: columns per pipeline block (MMA N)
constexpr int kExpandVCol = 2 * EBN;      // first TMEM column of V
constexpr int kExpandTmemCols = 256;      // 2 accumulators + V hi + V lo (rpad <= 128: 128 columns)

template <int DT>
__global__ void __launch_bounds__(EXP_THREADS, 2) tc_expand_kernel(const __grid_constant__ CUtensorMap tm_b,
                                                                const __grid_constant__ CUtensorMap tm_y,
                                                                const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const ExpandSmem L = ExpandSmem::make(p.rpad, p.bm, p.stages);
  const int EBUF = L.nbuf;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);  // [EBUF] y tile + B rows landed
  uint64_t *empty = full + MAX_EBUF;      // [EBUF] the buffer's y tile has been stored (or written)
  uint64_t *accfull = empty + MAX_EBUF;   // [2] accumulator a holds a finished block
  uint64_t *accempty = accfull + 2;   // [2] the epilogue has read accumulator a
  uint64_t *mmadone = accempty + 2;   // every MMA this CTA issued has completed
  uint64_t *ystaged = mmadone + 1;    // [EBUF] the epilogue has finished the buffer's y tile
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ystaged + MAX_EBUF);
  int32_t *flags = reinterpret_cast<int32_t *>(tmem_slot + 1);  // [0] = timed out
  TcTile *ti = reinterpret_cast<TcTile *>(smem + L.bar_off + 256);
  int32_t *scan = reinterpret_cast<int32_t *>(smem + L.bar_off + 1024);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y;
  const int nb_begin = blockIdx.x * p.nper;
  const int nb_end = min(nb_begin + p.nper, p.nblk_total);
  const int nblk = max(nb_end - nb_begin, 0);

  if (tid == 0) {
    for (int b = 0; b < EBUF; ++b) {
      mbar_init(&full[b], p.paged ? 1 + 32 : 1);  // paged: + one cp.async arrival per producer lane
      mbar_init(&empty[b], 1);
      mbar_init(&ystaged[b], EXP_EPI_WARPS * 32);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accfull[a], 1);
      mbar_init(&accempty[a], EXP_EPI_WARPS * 32);
    }
    mbar_init(mmadone, 1);
    flags[0] = 0;
    mbar_fence_init();
    tc::tma_prefetch_desc(&tm_b);
    tc::tma_prefetch_desc(&tm_y);
  }
  // tensor memory: two EBN-column accumulators, then V hi (rpad / 2 columns: two 16-bit elements
  // per column) and V lo; two CTAs per SM take all 512 columns
  if (warp == 0) tc::tmem_alloc(tmem_slot, kExpandTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  resolve_tc_tile(p, t, ti, scan);  // every thread; ends with a barrier
  int32_t *ptab = scan;               // paged: the scan area is free after the resolve
  bool active = !ti->skip && nblk > 0;
  int32_t bad = ti->bad;
  if (p.paged && active && load_page_ids(p, p.b_tab, p.b_ppv, ti->slot, ti->rank, ptab)) {
    bad |= MLORA_STATUS_BAD_PAGE;
    active = false;
  }
  const int row0 = ti->row0, nr = ti->nr, s = ti->slot, rank = ti->rank;
  const float scale = ti->scale;
  const bool full_tile = nr == p.bm;  // a partial tile writes its rows with plain stores: the
                                    // rows past nr belong to another segment
  const int brow = (s * p.num_layers + p.layer) * p.r_max;
  // bytes a block's TMA loads bring: the y tile, and the B rows unless they are gathered
  const uint32_t block_tx = (uint32_t)((p.paged ? 0 : p.rpad * 128) + p.bm * 128);
  const uint32_t idesc = tc::idesc_f16(DT == MLORA_BF16, false, true, BM, EBN);
  auto buf = [&](int i) { return smem + L.buf_off + (i % EBUF) * L.buf_bytes; };

  // producer: the first EBUF blocks go out before V is built
  int issued = 0;
  // one block's loads: lane 0 TMA-loads the y tile (and B rows of a stacked pool); for a paged
  // pool the whole producer warp gathers the B rows from their pages with cp.async
  auto issue = [&](int i) {
    uint8_t *dst = buf(i);
    const int nb = nb_begin + i;
    if (lane == 0) {
      mbar_arrive_expect_tx(&full[i % EBUF], block_tx);
      tc::tma_load_2d(dst, &tm_y, nb * EBN, row0, &full[i % EBUF]);
      if (!p.paged) tc::tma_load_2d(dst + L.b_in_buf, &tm_b, nb * EBN, brow, &full[i % EBUF]);
    }
    if (p.paged) {
      gather_atom(p, ptab, p.b_ppv, p.d_out, nb * EBN, dst + L.b_in_buf, lane);
      tc::cp_async_arrive(&full[i % EBUF]);
    }
  };
  if (active && warp == EXP_EPI_WARPS && (p.paged || lane == 0))
    for (; issued < nblk && issued < EBUF; ++issued) issue(issued);

  // Launched right behind the shrink of the same call (programmatic dependent launch), the kernel
  // has so far read only what that shrink does not write: metadata, page tables, B rows and the
  // y tiles (written, if at all, by work that completed before the shrink started). v and the
  // status word wait for the shrink's grid. Every CTA waits, so this grid never completes before
  // the shrink's.
  pdl_wait();
  if (blockIdx.x == 0 && tid == 0 && bad) report(p.status, bad);

  // V hi / lo in tensor memory (the MMA's A operand, K-major): thread m of warps 0-3 writes row m
  // (TMEM lane m), columns kExpandVCol + c hold elements 2c, 2c + 1 of V hi, and rpad / 2 columns
  // further those of V lo. fp16 rows are stored as v * 2^-vexp[m], with vexp[m] chosen so that the
  // row's largest |v| stays below 2^14 (fp16 overflows at 65504, where bf16 and the fp32 v do not);
  // the epilogue of row m multiplies its sums by 2^vexp[m]. The scaling is exact (a power of two);
  // bf16 rows are not scaled.
  int32_t *vexp = reinterpret_cast<int32_t *>(smem + L.bar_off + 512);  // [BM]
  if (active && warp < 4) {
    const int m = tid;
    const bool row_ok = m < nr;
    const float *vrow = p.v + (int64_t)(row0 + (row_ok ? m : 0)) * p.r_max;
    const bool vec = ((p.r_max & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.v) & 15) == 0);
    const int nc = p.rpad / 8;  // 8-element chunks of a row (at most 16)
    // Chunks g .. g + VG - 1 of row m (those below nc) into f, zero past the rank and for rows past
    // nr. A group inside the v row takes 2 VG loads of 16 bytes, all issued before any is used (the
    // row comes from L2: one round trip per group); otherwise single guarded floats. VG = 4 keeps
    // the kernel within the registers of two CTAs per SM.
    constexpr int VG = 4;
    auto load_group = [&](int g, float (&f)[VG][8]) {
      if (vec && (g + VG) * 8 <= p.r_max) {
#pragma unroll
        for (int u = 0; u < VG; ++u) {
          const float4 lo4 = *reinterpret_cast<const float4 *>(vrow + (g + u) * 8);
          const float4 hi4 = *reinterpret_cast<const float4 *>(vrow + (g + u) * 8 + 4);
          f[u][0] = lo4.x; f[u][1] = lo4.y; f[u][2] = lo4.z; f[u][3] = lo4.w;
          f[u][4] = hi4.x; f[u][5] = hi4.y; f[u][6] = hi4.z; f[u][7] = hi4.w;
        }
#pragma unroll
        for (int u = 0; u < VG; ++u)
#pragma unroll
          for (int e = 0; e < 8; ++e) f[u][e] = (row_ok && (g + u) * 8 + e < rank) ? f[u][e] : 0.f;
      } else {
#pragma unroll
        for (int u = 0; u < VG; ++u)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = (g + u) * 8 + e;
            f[u][e] = (row_ok && g + u < nc && j < rank) ? vrow[j] : 0.f;
          }
      }
    };
    float rs = 1.f;  // 2^-vexp[m]
    if constexpr (DT == MLORA_FP16) {
      float amax = 0.f;
      for (int g = 0; g < nc; g += VG) {
        float f[VG][8];
        load_group(g, f);
#pragma unroll
        for (int u = 0; u < VG; ++u)
#pragma unroll
          for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[u][e]));
      }
      int e2 = 0;
      (void)frexpf(amax, &e2);  // amax = mant * 2^e2, mant in [0.5, 1); e2 <= 128
      const int s = e2 > 14 ? e2 - 14 : 0;
      vexp[m] = s;
      rs = __int_as_float((127 - s) << 23);
    } else {
      vexp[m] = 0;
    }
    const uint32_t vrow_t = tmem + ((uint32_t)((warp & 3) * 32) << 16) + kExpandVCol;
    for (int g = 0; g < nc; g += VG) {
      float f[VG][8];
      load_group(g, f);
#pragma unroll
      for (int u = 0; u < VG; ++u) {
        if (g + u < nc) {  // 8 K elements = 4 TMEM columns
          float hi[8], lo[8];
          if constexpr (DT == MLORA_FP16) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[u][e] *= rs;
          }
          const uint4 h = pack8<DT>(f[u]);
          unpack8<DT>(h, hi);
#pragma unroll
          for (int e = 0; e < 8; ++e) lo[e] = f[u][e] - hi[e];
          const uint4 l = pack8<DT>(lo);
          tc::tmem_st4(vrow_t + (uint32_t)((g + u) * 4), h);
          tc::tmem_st4(vrow_t + (uint32_t)(p.rpad / 2 + (g + u) * 4), l);
        }
      }
    }
    tc::tmem_st_wait();
  }
  tc::tc_fence_before();
  __syncthreads();

  if (active && warp == EXP_EPI_WARPS) {
    // ---- producer (lane 0, or the whole warp for a paged pool): refill a buffer once its y
    // tile has been stored
    if (p.paged || lane == 0) {
      for (; issued < nblk; ++issued) {
        const int i = issued;
        const int ok = mbar_wait(&empty[i % EBUF], (uint32_t)((i / EBUF) - 1) & 1u) ? 1 : 0;
        if (p.paged ? __any_sync(0xffffffffu, !ok) : !ok) {
          if (lane == 0) flags[0] = 1;
          break;
        }
        issue(i);
      }
      // nothing may land in shared memory after the CTA exits: wait for the last loads (bounded)
      if (lane == 0)
        for (int i = max(issued - EBUF, 0); i < issued; ++i)
          (void)mbar_wait(&full[i % EBUF], (uint32_t)(i / EBUF) & 1u, kDrainLimitNs);
    }
    __syncwarp();
  } else if (active && warp == EXP_EPI_WARPS + 1) {
    // ---- MMA issuer (one lane)
    if (lane == 0) {
      int i = 0;
      for (; i < nblk; ++i) {
        const int a = i & 1;
        if (!mbar_wait(&full[i % EBUF], (uint32_t)(i / EBUF) & 1u) ||
            (i >= 2 && !mbar_wait(&accempty[a], (uint32_t)((i >> 1) - 1) & 1u))) {
          flags[0] = 1;
          break;
        }
        uint8_t *bs = buf(i) + L.b_in_buf;
        if (p.paged) tc::fence_proxy_async();  // the cp.async-gathered B rows -> the tensor cores
        if (rank < p.rpad) {  // rows rank..rpad-1 of B are padding (possibly NaN): zero them
          for (int e = 0; e < (p.rpad - rank) * 8; ++e)
            *reinterpret_cast<uint4 *>(bs + (rank + e / 8) * 128 + (e % 8) * 16) = make_uint4(0, 0, 0, 0);
          tc::fence_proxy_async();
        }
        tc::tc_fence_after();
        const int ksteps = p.rpad / 16;
        for (int part = 0; part < 2; ++part) {  // V hi, then V lo (from tensor memory)
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint32_t va = tmem + (uint32_t)(kExpandVCol + part * (p.rpad / 2) + kk * 8);  // 16 K elements
            const uint64_t db = tc::smem_desc_sw128(bs + kk * 16 * 128, 16, 1024);
            tc::mma_f16_tmem_a(tmem + (uint32_t)(a * EBN), va, db, idesc, (part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(&accfull[a]);
      }
      // every MMA issued so far completes before TMEM is released (bounded)
      tc::mma_commit(mmadone);
      (void)mbar_wait(mmadone, 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (active && warp == EXP_EPI_WARPS + 2) {
    // ---- store (one lane): each finished y tile goes out by TMA; its buffer is freed once the
    // store has read it (a partial tile was written by the epilogue with plain stores). One store
    // at a time: freeing a buffer a block later (two stores in flight) shortens the load ring,
    // and loads are what limits this kernel (7 expands of the 13B prefill 723 -> 834 us).
    if (lane == 0) {
      for (int i = 0; i < nblk; ++i) {
        if (!mbar_wait(&ystaged[i % EBUF], (uint32_t)(i / EBUF) & 1u)) {
          flags[0] = 1;
          break;
        }
        if (full_tile) {
          tc::tma_store_2d(&tm_y, (nb_begin + i) * EBN, row0, buf(i));  // columns past d_out are clipped
          tc::bulk_commit_group();
          tc::bulk_wait_group_read<0>();
        }
        mbar_arrive(&empty[i % EBUF]);
      }
      tc::bulk_wait_group_all();  // stores complete before the shared memory goes away
    }
    __syncwarp();
  } else if (active) {
    // ---- epilogue: row m of the block's y tile += scale * D (this warp's 32 columns), rounded once
    const int m = (warp & 3) * 32 + lane, half = warp >> 2;
    // fp16 V row m was stored scaled by 2^-vexp[m]: its sums carry the factor back (exact)
    const float rscale = DT == MLORA_FP16 ? scale * __int_as_float((127 + vexp[m]) << 23) : scale;
    int i = 0;
    for (; i < nblk; ++i) {
      const int a = i & 1, nb = nb_begin + i;
      uint8_t *ys = buf(i);
      int ok = mbar_wait(&accfull[a], (uint32_t)(i >> 1) & 1u) ? 1 : 0;
      ok &= mbar_wait(&full[i % EBUF], (uint32_t)(i / EBUF) & 1u) ? 1 : 0;  // the y tile is visible
      if (!ok) {  // no barrier across the epilogue warps: each goes its own pace; a thread that
                  // gives up leaves its later arrivals out, so the other roles' bounded waits end too
        flags[0] = 1;
        break;
      }
      tc::tc_fence_after();
      float d[EBN / 2];
#pragma unroll
      for (int c16 = 0; c16 < EBN / 32; ++c16) {
        float q[16];
        tc::tmem_ld16(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(a * EBN + half * (EBN / 2) + c16 * 16), q);
#pragma unroll
        for (int e = 0; e < 16; ++e) d[c16 * 16 + e] = q[e];
      }
      tc::tc_fence_before();
      mbar_arrive(&accempty[a]);  // the accumulator may take the block after next
      if (m < nr) {  // accumulator rows past the tile's rows (m >= nr, at most bm) are not the tile's
#pragma unroll
        for (int cq = 0; cq < EBN / 16; ++cq) {  // this warp's 16-byte chunks of the 128-byte row
          const int ch = half * (EBN / 16) + cq;
          uint4 *cell = reinterpret_cast<uint4 *>(ys + m * 128 + ((ch ^ (m & 7)) << 4));
          float yf[8];
          unpack8<DT>(*cell, yf);
#pragma unroll
          for (int e = 0; e < 8; ++e) yf[e] = fmaf(rscale, d[cq * 8 + e], yf[e]);
          if (full_tile) {
            *cell = pack8<DT>(yf);
          } else if (nb * EBN + ch * 8 < p.d_out) {
            *reinterpret_cast<uint4 *>(p.y + (int64_t)(row0 + m) * p.ldy + nb * EBN + ch * 8) = pack8<DT>(yf);
          }
        }
      }
      tc::fence_proxy_async();          // this thread's y writes -> visible to the TMA store
      mbar_arrive(&ystaged[i % EBUF]);  // the store warp takes the tile from here
    }
  }
  __syncthreads();
  if (active && flags[0] && tid == 0) report(p.status, MLORA_STATUS_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kExpandTmemCols);
}

// ------------------------------------------------------------------------------------------
// host

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// 2-D map over `rows` rows of `cols` 16-bit elements with a row pitch of `ld` elements;
// box = 64 columns x box_rows rows, 128-byte swizzle, zero fill outside the tensor.
bool encode_2d(CUtensorMap *m, int dtype, const void *base, int64_t cols, int64_t rows, int64_t ld, int box_rows) {
  EncodeFn fn = encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dtype == MLORA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename K>
cudaError_t set_smem(K kern, size_t smem) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

// Rows from which a segment runs on the tensor cores: kTcMinRows, lowered for a batch of few
// segments so that nseg * (tc_min - 1) -- the short-segment tiles the CUDA-core launch is sized
// for -- stays near the SM count; at least kTcMinRowsLow.
int tc_min_rows(int nseg) {
  const int t = 1 + sm_count() / (nseg > 0 ? nseg : 1);
  return t < kTcMinRowsLow ? kTcMinRowsLow : t > kTcMinRows ? kTcMinRows : t;
}

// The host does not see the segment lengths, only the batch's size: the tensor-core kernels are
// launched for a batch with enough rows for long segments to be worth two extra launches (at
// least kTcBatchRows rows, kTcAvgRows per segment on average -- a prefill batch, or prompts mixed
// with decode rows). They take every segment of at least kTcMinRows rows; the CUDA-core kernel
// takes the rest. A decode batch (a few rows per segment) runs on the CUDA-core kernel alone.
bool tc_eligible(const PoolDev &pool, int num_rows, int nseg) {
  const int rpad = (pool.r_max + 15) & ~15;
  // paged pools: pages of at least 64 elements (an atom crosses at most one page boundary), and
  // the page ids of a tile's vectors fit the table area of shared memory
  const bool paged_ok = pool.kind == MLORA_POOL_PAGED && pool.page_elems >= 64 &&
                        rpad * pool.a_ppv <= 2 * SCAN_CAP && rpad * pool.b_ppv <= 2 * SCAN_CAP;
  return (pool.kind == MLORA_POOL_STACKED || paged_ok) && (pool.dtype == MLORA_BF16 || pool.dtype == MLORA_FP16) &&
         pool.r_max <= 128 && num_rows >= kTcBatchRows &&
         (int64_t)num_rows >= (int64_t)kTcAvgRows * (nseg > 0 ? nseg : 1) && encoder() != nullptr;
}

// Rows per tile: chunks small enough that the tiles of the long segments fill the SMs in one wave
// (at most M / bm + nseg tiles), a multiple of 8 rows (the swizzle atom), between kMinTileRows
// and the MMA's 128.
int tile_rows(int M, int nseg) {
  const int avail = sm_count() - nseg;
  int bm = BM;
  if (avail > 0) bm = ((M + avail - 1) / avail + 7) & ~7;
  return bm < kMinTileRows ? kMinTileRows : bm > BM ? BM : bm;
}

cudaError_t launch_tc_shrink(const ProblemDev &pr, TcParams p, cudaStream_t stream) {
  const PoolDev &pl = pr.pool;
  p.rpad = (pl.r_max + 15) & ~15;
  p.tmem_cols = p.rpad <= 32 ? 32 : p.rpad <= 64 ? 64 : 128;
  p.bm = tile_rows(p.M, p.nseg);
  p.tiles = p.M / p.bm + p.nseg;  // >= sum over long segments of ceil(len / bm)
  if (p.tiles <= 0) return cudaSuccess;
  const int kb_total = (pl.d_in + SKA * BK - 1) / (SKA * BK);
  p.stages = ShrinkSmem::make(p.rpad, p.bm).stages;
  const size_t smem = ShrinkSmem::make(p.rpad, p.bm, p.stages).total;
  auto kern = pl.dtype == MLORA_BF16 ? tc_shrink_kernel<MLORA_BF16> : tc_shrink_kernel<MLORA_FP16>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  // K split: as many parts as keep the whole grid resident (one wave)
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NTHREADS, smem) != cudaSuccess || occ < 1) occ = 1;
  int ks = occ * sm_count() / (p.tiles > 0 ? p.tiles : 1);
  ks = ks < 1 ? 1 : ks > 4 ? 4 : ks;
  ks = ks > kb_total ? kb_total : ks;
  p.ksplit = ks;
  CUtensorMap tm_x, tm_a;
  if (!encode_2d(&tm_x, pl.dtype, pr.x, pl.d_in, p.M, pr.ldx, p.bm)) return cudaErrorInvalidValue;
  if (p.paged) {
    tm_a = tm_x;  // not read: the A^T rows are gathered from the pages
  } else if (!encode_2d(&tm_a, pl.dtype, pl.a_t, pl.d_in, (int64_t)pl.num_slots * pl.num_layers * pl.r_max, pl.d_in,
                        p.rpad)) {
    return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks, p.tiles, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_a, p);
}

cudaError_t launch_tc_expand(const ProblemDev &pr, TcParams p, cudaStream_t stream, bool after_shrink) {
  const PoolDev &pl = pr.pool;
  p.rpad = (pl.r_max + 15) & ~15;
  // Full 128-row tiles: the expand's cost per block is its y tile's pipeline pass, and tiles of
  // fewer rows measured slower (13B prefill, 7 expands: 689 us with 128 rows, 776 us with 88).
  p.bm = BM;
  p.tiles = p.M / p.bm + p.nseg;
  if (p.tiles <= 0) return cudaSuccess;
  p.nblk_total = (pl.d_out + EBN - 1) / EBN;
  // Column runs per tile: the grid is about two waves of the expand's two CTAs per SM (measured
  // best on the 13B prefill: 16 blocks of 64 columns per CTA at d_out 5120, ~40 at 13824;
  // shorter runs pay the V setup more often, longer ones leave SMs idle).
  {
    int runs = 4 * sm_count() / (p.tiles > 0 ? p.tiles : 1);
    runs = runs < 1 ? 1 : runs > p.nblk_total ? p.nblk_total : runs;
    p.nper = (p.nblk_total + runs - 1) / runs;
  }
  const int expand_budget = 112 * 1024;  // two CTAs per SM
  CUtensorMap tm_b, tm_y;
  if (!encode_2d(&tm_y, pl.dtype, pr.y, pl.d_out, p.M, pr.ldy, p.bm)) return cudaErrorInvalidValue;
  if (p.paged) {
    tm_b = tm_y;  // not read: the B rows are gathered from the pages
  } else if (!encode_2d(&tm_b, pl.dtype, pl.b, pl.d_out, (int64_t)pl.num_slots * pl.num_layers * pl.r_max, pl.d_out,
                        p.rpad)) {
    return cudaErrorInvalidValue;
  }
  p.stages = ExpandSmem::make(p.rpad, p.bm, 0, expand_budget).nbuf;
  const size_t smem = ExpandSmem::make(p.rpad, p.bm, p.stages).total;
  auto kern = pl.dtype == MLORA_BF16 ? tc_expand_kernel<MLORA_BF16> : tc_expand_kernel<MLORA_FP16>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.nblk_total + p.nper - 1) / p.nper, p.tiles, 1);
  cfg.blockDim = dim3(EXP_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // right behind the tensor-core shrink of the same call: start early (programmatic dependent
  // launch), the kernel waits for the shrink before it reads v
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_shrink ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tm_b, tm_y, p);
}

}  // namespace mlora
