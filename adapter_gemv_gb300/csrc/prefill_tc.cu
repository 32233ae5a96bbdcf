// prefill_tc.cu -- tensor-core path for long SGMV segments (prefill), sm_103a.
//
// A segment of L >= 128 rows that shares one adapter is a real dense contraction ("the segments
// are short and fat, so the work is closer to a GEMM", "Multi-LoRA Serving, in depth", section
// "Two shapes: SGMV for prefill, BGMV for decode"; Punica section 3.4, "Tensor Core usage"). Its
// full 128-row blocks run here; the ragged tail of each segment runs on the CUDA-core kernels.
//
//   shrink  V[128 x r] = X[128 x d_in] . A   : one CTA per (tile, K part); a cluster of K parts
//           sums its fp32 partials through distributed shared memory. X tiles and A^T rows are
//           both K-major; TMA (128-byte swizzle) feeds a 4-stage mbarrier ring, one thread issues
//           tcgen05.mma (M = 128, N = rank rounded up to 16, K = 16 per instruction) into a TMEM
//           accumulator, and all four warps read it back with tcgen05.ld.
//   expand  Y[128 x 128] += scale . V[128 x r] . B[r x 128] : one CTA per (tile, run of N blocks).
//           V (fp32) is split into bf16 hi + lo parts, so the product keeps ~16 bits of v, and
//           both parts are multiplied into one fp32 accumulator. B rows are an MN-major operand
//           loaded by TMA; y is read and written by the epilogue threads (one row each).
// Every wait is bounded; a timed-out CTA reports MLORA_STATUS_TIMEOUT and writes nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace mlora {

namespace {

constexpr int BM = 128;      // rows per tile (MMA M)
constexpr int BK = 64;       // K elements per stage (one 128-byte swizzle row)
constexpr int STAGES = 4;    // shrink ring depth
constexpr int BN = 128;      // expand: columns per N block (MMA N)
constexpr int NTHREADS = 128;
constexpr int SCAN_CAP = 512;

struct TcTile {
  int32_t row0, slot, rank, skip, bad;
  float scale;
};

// Tile t = the t-th full 128-row block, walking the segments in order (each contributes
// floor(len / 128) blocks). Whole block participates; row metadata only.
__device__ void resolve_tc_tile(const TcParams &p, int t, TcTile *ti, int32_t *scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    ti->skip = 1;
    ti->bad = 0;
  }
  __syncthreads();
  int32_t carry = 0, found = 0, bad = 0;
  for (int base = 0; base < p.nseg; base += SCAN_CAP) {
    const int cnt = min(SCAN_CAP, p.nseg - base);
    for (int q = tid; q <= cnt; q += NTHREADS) {
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
        const int32_t nt = (q < cnt && len > 0) ? len / BM : 0;
        int32_t incl = nt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += o;
        }
        const int32_t excl = carry + incl - nt;
        const bool mine = q < cnt && t >= excl && t < excl + nt;
        if (!found && mine) {
          ti->row0 = lo + (t - excl) * BM;
          ti->slot = scan[SCAN_CAP + 1 + q];
        }
        found |= __any_sync(0xffffffffu, mine);
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      bad = __any_sync(0xffffffffu, bad);
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
        const int r = p.rank[s];
        if (r < 1 || r > p.r_max) {
          b = MLORA_STATUS_BAD_RANK;
          skip = 1;
        } else {
          ti->rank = r;
          ti->scale = p.scale[s];
        }
      }
    }
    ti->bad = b;
    ti->skip = skip;
  }
  __syncthreads();
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------------------------------
// shrink

struct ShrinkSmem {
  int stage_bytes, a_off, bar_off, total;
  __host__ __device__ static ShrinkSmem make(int rpad) {
    ShrinkSmem L;
    L.a_off = BM * BK * 2;                                   // X tile: 16 KB
    L.stage_bytes = (L.a_off + rpad * BK * 2 + 1023) & ~1023;  // + A^T rows
    L.bar_off = STAGES * L.stage_bytes;
    L.total = L.bar_off + 1024 + (2 * SCAN_CAP + 1) * 4 + 1024;  // barriers, tile info, scan, alignment slack
    return L;
  }
};

template <int DT>
__global__ void __launch_bounds__(NTHREADS) tc_shrink_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                             const __grid_constant__ CUtensorMap tm_a,
                                                             const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const ShrinkSmem L = ShrinkSmem::make(p.rpad);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
  uint64_t *empty = full + STAGES;
  uint64_t *accbar = empty + STAGES;
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
      mbar_init(&full[s], 1);
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

  resolve_tc_tile(p, t, ti, scan);
  if (c == 0 && tid == 0 && ti->bad) report(p.status, ti->bad);
  const bool active = !ti->skip;
  const int row0 = ti->row0, s = ti->slot, rank = ti->rank;
  const int kb_total = (p.d_in + BK - 1) / BK;
  const int kb_per = (kb_total + ks - 1) / ks;
  const int kb0 = min((int)c * kb_per, kb_total), kb1 = min(kb0 + kb_per, kb_total);
  const int nkb = active ? kb1 - kb0 : 0;
  const int arow = (s * p.num_layers + p.layer) * p.r_max;
  const uint32_t stage_tx = (uint32_t)(BM * BK * 2 + p.rpad * BK * 2);
  const uint32_t idesc = tc::idesc_f16(DT == MLORA_BF16, false, false, BM, p.rpad);

  if (warp == 0) {
    // producer (one lane): TMA X tile and A^T rows of each K block into the ring
    for (int i = 0; lane == 0 && i < nkb; ++i) {
      const int st = i % STAGES;
      if (i >= STAGES && !mbar_wait(&empty[st], (uint32_t)((i / STAGES) - 1) & 1u)) {
        flags[0] = 1;
        break;
      }
      uint8_t *sb = smem + st * L.stage_bytes;
      mbar_arrive_expect_tx(&full[st], stage_tx);
      tc::tma_load_2d(sb, &tm_x, (kb0 + i) * BK, row0, &full[st]);
      tc::tma_load_2d(sb + L.a_off, &tm_a, (kb0 + i) * BK, arow, &full[st]);
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
      tc::tc_fence_after();
      const uint8_t *sb = smem + st * L.stage_bytes;
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        const uint64_t da = tc::smem_desc_sw128(sb + k * 32, 16, 1024);
        const uint64_t db = tc::smem_desc_sw128(sb + L.a_off + k * 32, 16, 1024);
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
  float *red = reinterpret_cast<float *>(smem);  // the ring is idle now: [128][rpad] fp32 partials
  const int m = warp * 32 + lane;
  if (active && !timed_out) {
    for (int c16 = 0; c16 < p.rpad / 16; ++c16) {
      float vals[16];
      if (nkb > 0) {
        tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c16 * 16), vals);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) vals[e] = 0.f;
      }
      if (ks == 1) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = c16 * 16 + e;
          if (j < rank) p.v[(int64_t)(row0 + m) * p.r_max + j] = vals[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) red[m * p.rpad + c16 * 16 + e] = vals[e];
      }
    }
  }
  if (ks > 1) {
    cluster_sync();
    if (active && !timed_out) {
      // CTA c sums rows [c * 128 / ks, (c + 1) * 128 / ks) over the cluster, in rank order
      const int rows_per = BM / ks;
      for (int e = tid; e < rows_per * rank; e += NTHREADS) {
        const int mm = (int)c * rows_per + e / rank, j = e % rank;
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

struct ExpandSmem {
  int v_off, b_off, b_buf, bar_off, total;
  __host__ __device__ static ExpandSmem make(int rpad) {
    ExpandSmem L;
    const int katoms = (rpad + BK - 1) / BK;
    L.v_off = 0;                                     // V hi, V lo: [2][katoms][128 rows x 128 B]
    L.b_off = 2 * katoms * BM * 128;
    L.b_buf = 2 * rpad * 128;                        // one N block: 2 MN atoms x rpad K rows x 128 B
    L.bar_off = L.b_off + 2 * ((L.b_buf + 1023) & ~1023);
    L.total = L.bar_off + 1024 + (2 * SCAN_CAP + 1) * 4 + 1024;
    return L;
  }
};

template <int DT>
__global__ void __launch_bounds__(NTHREADS) tc_expand_kernel(const __grid_constant__ CUtensorMap tm_b,
                                                             const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const ExpandSmem L = ExpandSmem::make(p.rpad);
  const int katoms = (p.rpad + BK - 1) / BK;
  const int bbuf = (L.b_buf + 1023) & ~1023;
  uint64_t *bfull = reinterpret_cast<uint64_t *>(smem + L.bar_off);  // [2]
  uint64_t *accbar = bfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accbar + 1);
  TcTile *ti = reinterpret_cast<TcTile *>(smem + L.bar_off + 256);
  int32_t *scan = reinterpret_cast<int32_t *>(smem + L.bar_off + 1024);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.y;
  const int nb_begin = blockIdx.x * p.nper;
  const int nb_end = min(nb_begin + p.nper, p.nblk_total);

  if (tid == 0) {
    mbar_init(&bfull[0], 1);
    mbar_init(&bfull[1], 1);
    mbar_init(accbar, 1);
    mbar_fence_init();
    tc::tma_prefetch_desc(&tm_b);
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, BN);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  resolve_tc_tile(p, t, ti, scan);
  if (blockIdx.x == 0 && tid == 0 && ti->bad) report(p.status, ti->bad);
  const bool active = !ti->skip && nb_begin < nb_end;
  const int row0 = ti->row0, s = ti->slot, rank = ti->rank;
  const float scale = ti->scale;
  const int brow = (s * p.num_layers + p.layer) * p.r_max;
  const uint32_t block_tx = (uint32_t)(2 * p.rpad * 128);
  const uint32_t idesc = tc::idesc_f16(DT == MLORA_BF16, false, true, BM, BN);
  int timed_out = 0;

  auto issue_b = [&](int nb) {  // both 64-column MN atoms of N block nb
    uint8_t *dst = smem + L.b_off + (nb & 1) * bbuf;
    mbar_arrive_expect_tx(&bfull[nb & 1], block_tx);
    tc::tma_load_2d(dst, &tm_b, nb * BN, brow, &bfull[nb & 1]);
    tc::tma_load_2d(dst + p.rpad * 128, &tm_b, nb * BN + 64, brow, &bfull[nb & 1]);
  };

  if (active) {
    if (warp == 0) {
      if (lane == 0) {
        issue_b(nb_begin);
        if (nb_begin + 1 < nb_end) issue_b(nb_begin + 1);
      }
      __syncwarp();
    }
    // V hi / lo in the K-major 128-byte-swizzle layout: thread m owns row m
    const int m = tid;
    const float *vrow = p.v + (int64_t)(row0 + m) * p.r_max;
    for (int c8 = 0; c8 < katoms * 8; ++c8) {  // 16-byte chunks of 8 K elements
      float f[8], hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = c8 * 8 + e;
        f[e] = (j < rank) ? vrow[j] : 0.f;
      }
      const uint4 h = pack8<DT>(f);
      unpack8<DT>(h, hi);
#pragma unroll
      for (int e = 0; e < 8; ++e) lo[e] = f[e] - hi[e];
      const uint4 l = pack8<DT>(lo);
      const int atom = c8 >> 3, ch = c8 & 7;
      const int off = atom * (BM * 128) + m * 128 + ((ch ^ (m & 7)) << 4);
      *reinterpret_cast<uint4 *>(smem + L.v_off + off) = h;
      *reinterpret_cast<uint4 *>(smem + L.v_off + katoms * BM * 128 + off) = l;
    }
    tc::fence_proxy_async();
  }
  __syncthreads();

  for (int nb = nb_begin; active && nb < nb_end && !timed_out; ++nb) {
    const int buf = nb & 1;
    uint8_t *bsm = smem + L.b_off + buf * bbuf;
    const int okb = mbar_wait(&bfull[buf], (uint32_t)((nb - nb_begin) >> 1) & 1u) ? 1 : 0;
    timed_out = __syncthreads_or(!okb);
    if (timed_out) break;
    if (rank < p.rpad) {
      // rows rank..rpad-1 of B are padding (possibly NaN): zero them in both MN atoms
      for (int e = tid; e < 2 * (p.rpad - rank) * 8; e += NTHREADS) {
        const int atom = e / ((p.rpad - rank) * 8), rem = e % ((p.rpad - rank) * 8);
        const int j = rank + rem / 8, ch = rem % 8;
        *reinterpret_cast<uint4 *>(bsm + atom * p.rpad * 128 + j * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async();
      __syncthreads();
    }
    if (warp == 1) {
      if (lane == 0) {
      tc::tc_fence_after();
      const int ksteps = p.rpad / 16;
      for (int part = 0; part < 2; ++part) {  // V hi, then V lo
        for (int kk = 0; kk < ksteps; ++kk) {
          const uint8_t *va = smem + L.v_off + part * katoms * BM * 128 + (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          const uint64_t da = tc::smem_desc_sw128(va, 16, 1024);
          const uint64_t db = tc::smem_desc_sw128(bsm + kk * 16 * 128, (uint32_t)(p.rpad * 128), 1024);
          tc::mma_f16(tmem, da, db, idesc, (part > 0 || kk > 0) ? 1u : 0u);
        }
      }
      tc::mma_commit(accbar);
      }
      __syncwarp();
    }
    // y of this thread's row for the block, requested while the MMAs run
    const int m = tid, n0 = nb * BN;
    uint16_t *yrow = p.y + (int64_t)(row0 + m) * p.ldy;
    uint4 yv[BN / 8];
#pragma unroll
    for (int q = 0; q < BN / 8; ++q)
      if (n0 + q * 8 < p.d_out) yv[q] = ldg_u4(yrow + n0 + q * 8);
    const int oka = mbar_wait(accbar, (uint32_t)(nb - nb_begin) & 1u) ? 1 : 0;
    timed_out = __syncthreads_or(!oka);
    if (timed_out) break;
    tc::tc_fence_after();
    if (warp == 0) {
      if (lane == 0 && nb + 2 < nb_end) issue_b(nb + 2);  // the MMAs are done with this buffer
      __syncwarp();
    }
#pragma unroll
    for (int c16 = 0; c16 < BN / 16; ++c16) {
      float d[16];
      tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c16 * 16), d);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = c16 * 2 + h;
        if (n0 + q * 8 < p.d_out) {
          float yf[8];
          unpack8<DT>(yv[q], yf);
#pragma unroll
          for (int e = 0; e < 8; ++e) yf[e] = fmaf(scale, d[h * 8 + e], yf[e]);
          *reinterpret_cast<uint4 *>(yrow + n0 + q * 8) = pack8<DT>(yf);
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();  // TMEM and the B buffer are reused by the next block
  }
  if (timed_out) {
    // copies still in flight land before the shared memory is released
    (void)mbar_wait(&bfull[0], 0, 100000000ull);
    if (tid == 0) report(p.status, MLORA_STATUS_TIMEOUT);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, BN);
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

int sm_count_tc() {
  static int n = 0;
  if (!n) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    n = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 148;
  }
  return n;
}

template <typename K>
cudaError_t set_smem(K kern, size_t smem) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

bool tc_eligible(const PoolDev &pool, int num_rows, int nseg) {
  return pool.kind == MLORA_POOL_STACKED && pool.dtype == MLORA_BF16 && pool.r_max <= 128 && num_rows >= BM &&
         (int64_t)num_rows >= (int64_t)64 * (nseg > 0 ? nseg : 1) && encoder() != nullptr;
}

cudaError_t launch_tc_shrink(const ProblemDev &pr, TcParams p, cudaStream_t stream) {
  const PoolDev &pl = pr.pool;
  p.rpad = (pl.r_max + 15) & ~15;
  p.tmem_cols = p.rpad <= 32 ? 32 : p.rpad <= 64 ? 64 : 128;
  p.tiles = p.M / BM;
  if (p.tiles <= 0) return cudaSuccess;
  const int kb_total = (pl.d_in + BK - 1) / BK;
  int ks = sm_count_tc() / p.tiles;
  ks = ks < 1 ? 1 : ks > 4 ? 4 : ks;
  ks = ks > kb_total ? kb_total : ks;
  p.ksplit = ks;
  CUtensorMap tm_x, tm_a;
  if (!encode_2d(&tm_x, pl.dtype, pr.x, pl.d_in, p.M, pr.ldx, BM)) return cudaErrorInvalidValue;
  if (!encode_2d(&tm_a, pl.dtype, pl.a_t, pl.d_in, (int64_t)pl.num_slots * pl.num_layers * pl.r_max, pl.d_in, p.rpad))
    return cudaErrorInvalidValue;
  const size_t smem = ShrinkSmem::make(p.rpad).total;
  auto kern = tc_shrink_kernel<MLORA_BF16>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
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

cudaError_t launch_tc_expand(const ProblemDev &pr, TcParams p, cudaStream_t stream) {
  const PoolDev &pl = pr.pool;
  p.rpad = (pl.r_max + 15) & ~15;
  p.tiles = p.M / BM;
  if (p.tiles <= 0) return cudaSuccess;
  p.nblk_total = (pl.d_out + BN - 1) / BN;
  p.nper = 4;
  CUtensorMap tm_b;
  if (!encode_2d(&tm_b, pl.dtype, pl.b, pl.d_out, (int64_t)pl.num_slots * pl.num_layers * pl.r_max, pl.d_out, p.rpad))
    return cudaErrorInvalidValue;
  const size_t smem = ExpandSmem::make(p.rpad).total;
  auto kern = tc_expand_kernel<MLORA_BF16>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.nblk_total + p.nper - 1) / p.nper, p.tiles, 1);
  kern<<<grid, NTHREADS, smem, stream>>>(tm_b, p);
  return cudaGetLastError();
}

}  // namespace mlora
