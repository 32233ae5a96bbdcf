// bgmv_plan.cu -- device-side grouping of BGMV rows (sm_103a).
//
// A decode batch in BGMV form lists a slot per row, in request order ("Multi-LoRA Serving, in
// depth", section "The decode cost model": a good kernel reads each adapter once per step).
// Punica's batch layout (section 3.4, "Batch Layout Construction") groups the rows that share an
// adapter into one segment before the kernels run. This kernel does that grouping on the GPU, so
// the caller's row order is kept: it writes an order of the rows, in which
//   * rows with the same slot are adjacent: their CTAs run at the same time and the adapter rows
//     come from HBM once (the later requests are served by L2 while the first is in flight);
//   * rows of higher rank come first (the rank is the work of a row: a rank-64 row moves eight
//     times the bytes of a rank-8 row), so the longest CTAs start in the first wave and the short
//     ones fill in behind them -- longest-first scheduling shortens the launch's tail;
//   * rows without adapter and rows with an invalid slot come last (the CUDA-core kernel skips
//     the first and reports the second).
// Key of row i: (r_max - rank[slot], slot, i), sorted by a bitonic network in shared memory (one
// CTA; the key holds the row index, so the order is unique and the same on every call).
// For the streaming kernel (bgmv_stream.cu) the order is also cut into segments: runs of rows that
// share a slot, at most seg_rows rows each (segs[0] = their count, segs[1 + k] = segment k's first
// position in the order). A segment's rows read their adapter's rank-rows once.
// Before griddepcontrol.wait the kernel reads only the rows' slots and the pool's rank table; the
// order (perm[t] = row, sslot[t] = its slot) and the segments are written after the wait, into
// caller-owned memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace mlora {

namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) bgmv_plan_kernel(const int32_t *__restrict__ row_slot, int32_t M,
                                                                 int32_t n2, const int32_t *__restrict__ rank,
                                                                 int32_t num_slots, int32_t r_max, int32_t *perm,
                                                                 int32_t *sslot, int32_t *segs, int32_t seg_rows) {
  extern __shared__ uint64_t keys[];  // [n2], then (segments) an int scratch [n2]
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    uint64_t key = ~0ull;  // padding past M sorts last
    if (i < M) {
      const int32_t s = row_slot[i];
      uint32_t rk = 255u;  // no adapter / invalid slot / invalid rank: last
      if (s >= 0 && s < num_slots) {
        const int32_t r = rank[s];
        if (r >= 1 && r <= r_max) rk = (uint32_t)(r_max - r);
      }
      key = ((uint64_t)rk << 56) | ((uint64_t)((uint32_t)s + 1u) << 16) | (uint64_t)i;
    }
    keys[i] = key;
  }
  __syncthreads();
  // bitonic sort, ascending
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int partner = i ^ stride;
        if (partner > i) {
          const bool ascending = (i & size) == 0;
          const uint64_t a = keys[i], b = keys[partner];
          if ((a > b) == ascending) {
            keys[i] = b;
            keys[partner] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  pdl_wait();  // the previous kernel may still be reading perm / sslot (the caller's scratch)
  for (int t = threadIdx.x; t < M; t += blockDim.x) {
    const uint64_t key = keys[t];
    perm[t] = (int32_t)(key & 0xFFFFu);
    sslot[t] = (int32_t)((uint32_t)(key >> 16) - 1u);
  }
  if (segs == nullptr) return;
  // Segments: the start of each run of equal (rank key, slot), by an inclusive max-scan; then a
  // segment every seg_rows rows of a run, compacted by an inclusive sum-scan. n2 <= 4096 and
  // blockDim = min(n2, 1024), so a thread holds at most 4 entries.
  int32_t *sc = reinterpret_cast<int32_t *>(keys + n2);
  const int bd = blockDim.x, tid = threadIdx.x;
  int32_t v[4];
  for (int k = 0; k < 4; ++k) {
    const int t = tid + k * bd;
    if (t < n2) sc[t] = (t < M && (t == 0 || (keys[t - 1] >> 16) != (keys[t] >> 16))) ? t : 0;
  }
  __syncthreads();
  for (int d = 1; d < n2; d <<= 1) {
    for (int k = 0; k < 4; ++k) {
      const int t = tid + k * bd;
      v[k] = (t < n2 && t >= d) ? sc[t - d] : 0;
    }
    __syncthreads();
    for (int k = 0; k < 4; ++k) {
      const int t = tid + k * bd;
      if (t < n2 && v[k] > sc[t]) sc[t] = v[k];
    }
    __syncthreads();
  }
  for (int k = 0; k < 4; ++k) {  // sc[t]: the start of t's run -> 1 where a segment starts
    const int t = tid + k * bd;
    v[k] = (t < M && (t - sc[t]) % seg_rows == 0) ? 1 : 0;
  }
  __syncthreads();
  for (int k = 0; k < 4; ++k) {
    const int t = tid + k * bd;
    if (t < n2) sc[t] = v[k];
  }
  __syncthreads();
  for (int d = 1; d < n2; d <<= 1) {
    for (int k = 0; k < 4; ++k) {
      const int t = tid + k * bd;
      v[k] = (t < n2 && t >= d) ? sc[t - d] : 0;
    }
    __syncthreads();
    for (int k = 0; k < 4; ++k) {
      const int t = tid + k * bd;
      if (t < n2) sc[t] += v[k];
    }
    __syncthreads();
  }
  for (int t = tid; t < M; t += bd)
    if (sc[t] != (t > 0 ? sc[t - 1] : 0)) segs[sc[t]] = t;  // segment sc[t] - 1 starts at t
  if (tid == 0) segs[0] = M > 0 ? sc[M - 1] : 0;
}

}  // namespace

cudaError_t launch_bgmv_plan(const int32_t *row_slot, int32_t M, const PoolDev &pool, int32_t *perm, int32_t *sslot,
                             int32_t *segs, int32_t seg_rows, cudaStream_t stream, bool pdl) {
  int32_t n2 = 1;
  while (n2 < M) n2 <<= 1;
  if (n2 > kPlanMaxRows || (segs != nullptr && seg_rows < 1)) return cudaErrorInvalidValue;
  const size_t smem = (size_t)n2 * (sizeof(uint64_t) + (segs != nullptr ? sizeof(int32_t) : 0));
  cudaError_t e = cudaFuncSetAttribute(bgmv_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(n2 < kPlanThreads ? (n2 < 32 ? 32 : n2) : kPlanThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, bgmv_plan_kernel, row_slot, M, n2, pool.rank, pool.num_slots, pool.r_max, perm,
                            sslot, segs, seg_rows);
}

}  // namespace mlora
