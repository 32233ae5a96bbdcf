// decode_launch.cu -- host side of the decode kernels: rows per tile, split, stage sizes, grid.
#include <cuda_runtime.h>

#include "decode_impl.cuh"
#include "launch.h"

namespace mlora {

namespace {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Split a chunk of `chunk` elements into equal blocks of at most `cap` elements, multiples of 8.
int balanced_block(int chunk, int cap) {
  cap = cap < 8 ? 8 : (cap & ~7);
  const int nblk = (chunk + cap - 1) / cap;
  return (((chunk + nblk - 1) / nblk) + 7) & ~7;
}

}  // namespace

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
  // adapters, BGMV), else 8 (4 above rank 64) so an adapter row is reused across rows.
  const bool sgmv = p.seg_off != nullptr;
  const bool multi = sgmv && p.M >= 2 * (p.nseg > 0 ? p.nseg : 1);
  p.rt = multi ? (r_alloc <= 64 ? 8 : 4) : 1;
  const int64_t tiles = !sgmv ? (int64_t)p.M : (p.rt == 1 ? (int64_t)p.M : (int64_t)p.nseg + (p.M + p.rt - 1) / p.rt);
  if (tiles <= 0) return cudaSuccess;
  p.tiles = (int32_t)tiles;
  const int64_t units = tiles * p.nprob;

  // CTAs per tile: aim at two resident CTAs per SM over the whole launch, at least 128
  // elements of the split dimension per CTA, at most 16 (a non-portable cluster above 8).
  const int target = 2 * sm_count();
  int cs = (int)((target + units - 1) / units);
  const int split_dim = (mode == MODE_EXPAND) ? d_out_max : d_in_max;
  const int max_cs = split_dim / 128 > 1 ? split_dim / 128 : 1;
  cs = cs < 1 ? 1 : cs;
  cs = cs > max_cs ? max_cs : cs;
  if (mode != MODE_EXPAND) cs = cs > (units * 8 >= target ? 8 : decode::MAX_CS) ? (units * 8 >= target ? 8 : decode::MAX_CS) : cs;
  if (force_csplit > 0) cs = force_csplit;
  p.csplit = cs;

  const int kchunk = ((d_in_max + cs - 1) / cs + 7) & ~7;
  const int nchunk = ((d_out_max + cs - 1) / cs + 7) & ~7;
  const int row_cap = (40 * 1024) / ((r_alloc + p.rt) * 2);  // elements per row in one stage
  p.kb = (mode == MODE_EXPAND) ? 8 : balanced_block(kchunk, row_cap);
  p.nb = (mode == MODE_SHRINK) ? 8 : balanced_block(nchunk, row_cap);
  p.sk = (mode == MODE_EXPAND) ? 1 : ((kchunk + p.kb - 1) / p.kb < decode::MAX_STAGES ? (kchunk + p.kb - 1) / p.kb : decode::MAX_STAGES);
  p.se = (mode == MODE_SHRINK) ? 1 : ((nchunk + p.nb - 1) / p.nb < decode::MAX_STAGES ? (nchunk + p.nb - 1) / p.nb : decode::MAX_STAGES);
  if (mode == MODE_EXPAND) p.sk = 0;
  if (mode == MODE_SHRINK) p.se = 0;
  const int gcs = (mode == MODE_EXPAND) ? 1 : cs;
  Layout L = Layout::make(gcs, p.rt, r_alloc, p.sk, p.kb, p.se, p.nb);
  while (L.total > 227 * 1024 && (p.sk > 1 || p.se > 1)) {
    if (p.sk >= p.se && p.sk > 1) --p.sk;
    else --p.se;
    L = Layout::make(gcs, p.rt, r_alloc, p.sk, p.kb, p.se, p.nb);
  }
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
