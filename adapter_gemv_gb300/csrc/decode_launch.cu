// decode_launch.cu -- host side of the decode kernels: rows per tile, split, stage sizes, grid.
#include <cuda_runtime.h>

#include <atomic>

#include "decode_impl.cuh"
#include "launch.h"

namespace mlora {

namespace {

int query_sm_count(int dev) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  return n;
}

}  // namespace

int sm_count() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  if (dev >= kMaxDevices) return query_sm_count(dev);
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {  // concurrent first calls store the same value
    n = query_sm_count(dev);
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t launch_decode(int mode, int dtype, DecodeParams p, cudaStream_t stream, bool pdl, int force_csplit) {
  using decode::Layout;
  int r_alloc = 1, d_in_max = 8, d_out_max = 8;
  for (int q = 0; q < p.nprob; ++q) {
    r_alloc = r_alloc > p.prob[q].pool.r_max ? r_alloc : p.prob[q].pool.r_max;
    d_in_max = d_in_max > p.prob[q].pool.d_in ? d_in_max : p.prob[q].pool.d_in;
    d_out_max = d_out_max > p.prob[q].pool.d_out ? d_out_max : p.prob[q].pool.d_out;
  }
  p.r_alloc = r_alloc;
  // Rows per tile: one row when the segments are a row or two long (decode with distinct
  // adapters, BGMV), else 4 (an adapter row is reused across 4 rows; measured faster than 8 on
  // decode steps, whose longer tiles cost more registers and more empty rows).
  const bool sgmv = p.seg_off != nullptr;
  // When the tensor-core kernels take the long segments (a prefill or mixed batch), the segments
  // left here are short -- in a mixed batch, the one-row segments of decode requests -- so the
  // batch's average segment length says nothing about them: one-row tiles.
  bool tc_split = false;
  for (int q = 0; q < p.nprob; ++q) tc_split |= p.prob[q].tc_min > 0;
  const bool multi = sgmv && !tc_split && p.M >= 2 * (p.nseg > 0 ? p.nseg : 1);
  p.rt = multi ? 4 : 1;
  const int64_t all_tiles =
      !sgmv ? (int64_t)p.M : (p.rt == 1 ? (int64_t)p.M : (int64_t)p.nseg + (p.M + p.rt - 1) / p.rt);
  int64_t tiles = 0;  // the most any problem has (virtual tiles past a problem's own count idle)
  for (int q = 0; q < p.nprob; ++q) {
    int64_t tq = all_tiles;
    const int tcm = p.prob[q].tc_min;
    if (sgmv && tcm > 0) {
      // only segments shorter than tc_min rows are left for these kernels
      const int64_t per_seg = (tcm - 1 + p.rt - 1) / p.rt;
      tq = tq < (int64_t)p.nseg * per_seg ? tq : (int64_t)p.nseg * per_seg;
    }
    tiles = tiles > tq ? tiles : tq;
  }
  if (tiles <= 0) return cudaSuccess;
  p.tiles = (int32_t)tiles;
  const int64_t units = tiles * p.nprob;

  // Rank rows per warp -> K elements per pass of A loads into registers.
  const int jpw = r_alloc <= 16 ? 2 : r_alloc <= 32 ? 4 : r_alloc <= 64 ? 8 : 16;
  const int kb = 256 * (16 / jpw);
  // CTAs per tile (cs): the smallest split whose CTA slice of d_in is one pass of A loads and
  // whose slice of B fits in 88 KB of shared memory (so two CTAs fit on an SM), raised until
  // the launch has at least a third (chained calls) or half as many CTAs as there are SMs; at least 256 elements of the
  // split dimension per CTA; at most 16 per cluster. Fewer, fuller CTAs leave SM room for the
  // next launch's CTAs (programmatic dependent launch) to start and fetch their adapter rows
  // while this one runs.
  const int sms = sm_count();
  const int b_cap = 88 * 1024;
  const int y_cap = 16 * 1024, y_total_cap = 110 * 1024;
  int cs_min = 1;
  if (mode != MODE_EXPAND) cs_min = (d_in_max + kb - 1) / kb;
  if (mode != MODE_SHRINK) {
    const int need = (int)(((int64_t)r_alloc * d_out_max * 2 + b_cap - 1) / b_cap);
    cs_min = cs_min > need ? cs_min : need;
  }
  if (p.rt > 1 && mode != MODE_SHRINK) {  // one pass of the expand loop per thread
    const int need = (d_out_max + 8 * decode::NTHREADS - 1) / (8 * decode::NTHREADS);
    cs_min = cs_min > need ? cs_min : need;
  }
  // ... but no split that makes the grid more than about four waves of resident CTAs (two per
  // SM): past that, CTAs that loop over several passes of A beat more, shorter CTAs
  // (Llama-2-70B q_proj, rank 64, 256 rows: 16 CTAs per row 211 us, 4 CTAs per row 120 us).
  const int64_t cs_cap = (8 * (int64_t)sms) / units;
  if (cs_min > cs_cap) cs_min = cs_cap > 1 ? (int)cs_cap : 1;
  // Chained calls (programmatic dependent launch) want fewer CTAs, so the next launch finds SM
  // room early; a call on its own wants more, to hide its latency.
  const int floor_ctas = pdl ? sms / 3 : sms / 2;
  int cs = (int)((floor_ctas + units - 1) / units);
  cs = cs > cs_min ? cs : cs_min;
  const int split_dim = (mode == MODE_EXPAND) ? d_out_max : d_in_max;
  const int max_cs = split_dim / 256 > 1 ? split_dim / 256 : 1;
  cs = cs > max_cs ? max_cs : cs;
  if (mode != MODE_EXPAND && cs > decode::MAX_CS) cs = decode::MAX_CS;
  cs = cs < 1 ? 1 : cs;
  if (force_csplit > 0) cs = force_csplit;
  p.csplit = cs;

  // B rows of the CTA's d_out slice go to shared memory when they fit.
  const int nchunk = ((d_out_max + cs - 1) / cs + 7) & ~7;
  p.nb = (mode != MODE_SHRINK && (int64_t)r_alloc * nchunk * 2 <= b_cap) ? nchunk : 0;
  p.kb = kb;
  // The x row of a one-row tile whose d_in slice spans several passes of A goes to shared
  // memory whole, when it fits in 32 KB; each pass then reads its part there.
  {
    const int kchunk = ((d_in_max + cs - 1) / cs + 7) & ~7;
    const int npass = (kchunk + kb - 1) / kb;
    p.xw = (mode != MODE_EXPAND && p.rt == 1 && npass > 1 && npass * kb * 2 <= 32 * 1024) ? npass * kb : 0;
  }
  // Paged pools: the resolve reads every page id of the tile's vectors (to check them); they stay
  // in shared memory for the address of every later load when they fit 8 KB (else the loads
  // read the table in global memory, one dependent round trip each time).
  p.npt = 0;
  for (int q = 0; q < p.nprob; ++q) {
    const PoolDev &pl = p.prob[q].pool;
    if (pl.kind == MLORA_POOL_PAGED) {
      const int need = pl.r_max * (pl.a_ppv + pl.b_ppv);
      p.npt = p.npt > need ? p.npt : need;
    }
  }
  if (p.npt > 2048) p.npt = 0;
  // The tile's y rows also go to shared memory, if the CTA stays small enough to share an SM
  // with another.
  const int lcs = (mode == MODE_EXPAND) ? 1 : cs;
  p.ny = 0;
  if (mode != MODE_SHRINK && p.rt * nchunk * 2 <= y_cap &&
      Layout::make(lcs, p.rt, r_alloc, kb, p.nb, nchunk, p.xw, p.npt).total <= y_total_cap)
    p.ny = nchunk;
  const Layout L = Layout::make(lcs, p.rt, r_alloc, kb, p.nb, p.ny, p.xw, p.npt);
  if (L.total > 227 * 1024) return cudaErrorInvalidConfiguration;

  const int64_t grid = units * cs;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int cluster = (mode == MODE_EXPAND) ? 1 : cs;
  switch (mode) {
    case MODE_SHRINK: return launch_decode_shrink(dtype, p, (unsigned)grid, L.total, cluster, pdl, stream);
    case MODE_EXPAND: return launch_decode_expand(dtype, p, (unsigned)grid, L.total, cluster, pdl, stream);
    default: return launch_decode_fused(dtype, p, (unsigned)grid, L.total, cluster, pdl, stream);
  }
}

}  // namespace mlora
