// common.cuh -- device helpers shared by the libmlora kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement primitives the kernels are built on:
// mbarriers with transaction counts, 1-D bulk copies (cp.async.bulk, the TMA engine's
// untiled form), thread-block-cluster barriers and distributed shared memory.
// Every wait here is bounded: it gives up after a time limit and reports it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "launch.h"
#include "mlora.h"

namespace mlora {

// ---- element types --------------------------------------------------------------------------

template <int DT>
struct Elem;
template <>
struct Elem<MLORA_BF16> {
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
  static __device__ __forceinline__ uint16_t from_float(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
};
template <>
struct Elem<MLORA_FP16> {
  static __device__ __forceinline__ float lo(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)w)); }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __half2float(__ushort_as_half((uint16_t)(w >> 16)));
  }
  static __device__ __forceinline__ uint16_t from_float(float f) { return __half_as_ushort(__float2half_rn(f)); }
};

// 8 packed 16-bit elements -> 8 floats
template <int DT>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
  f[0] = Elem<DT>::lo(u.x); f[1] = Elem<DT>::hi(u.x);
  f[2] = Elem<DT>::lo(u.y); f[3] = Elem<DT>::hi(u.y);
  f[4] = Elem<DT>::lo(u.z); f[5] = Elem<DT>::hi(u.z);
  f[6] = Elem<DT>::lo(u.w); f[7] = Elem<DT>::hi(u.w);
}

// 8 packed 16-bit elements -> 4 float pairs, for the paired fp32 FMA (__ffma2_rn)
template <int DT>
__device__ __forceinline__ void unpack8x2(const uint4 &u, float2 (&f)[4]) {
  f[0] = make_float2(Elem<DT>::lo(u.x), Elem<DT>::hi(u.x));
  f[1] = make_float2(Elem<DT>::lo(u.y), Elem<DT>::hi(u.y));
  f[2] = make_float2(Elem<DT>::lo(u.z), Elem<DT>::hi(u.z));
  f[3] = make_float2(Elem<DT>::lo(u.w), Elem<DT>::hi(u.w));
}

// Mixed-precision FMA on packed 16-bit pairs: c0 += lo(x) * lo(a), c1 += hi(x) * hi(a), with
// 16-bit operands and fp32 accumulators, one instruction per product and no unpacking. Like the
// fp32 FMA on the unpacked operands, each computes x * a + c and rounds once, so the results
// are the same.
template <int DT>
__device__ __forceinline__ void mfma2(uint32_t x, uint32_t a, float &c0, float &c1) {
  if constexpr (DT == MLORA_BF16)
    asm("{ .reg .b16 xl, xh, al, ah; mov.b32 {xl, xh}, %2; mov.b32 {al, ah}, %3;\n"
        " fma.rn.f32.bf16 %0, xl, al, %0; fma.rn.f32.bf16 %1, xh, ah, %1; }"
        : "+f"(c0), "+f"(c1) : "r"(x), "r"(a));
  else
    asm("{ .reg .b16 xl, xh, al, ah; mov.b32 {xl, xh}, %2; mov.b32 {al, ah}, %3;\n"
        " fma.rn.f32.f16 %0, xl, al, %0; fma.rn.f32.f16 %1, xh, ah, %1; }"
        : "+f"(c0), "+f"(c1) : "r"(x), "r"(a));
}
// Eight products of chunk xv with chunk av (8 packed elements each) into the chains c0, c1.
template <int DT>
__device__ __forceinline__ void mfma8(const uint4 &xv, const uint4 &av, float &c0, float &c1) {
  mfma2<DT>(xv.x, av.x, c0, c1);
  mfma2<DT>(xv.y, av.y, c0, c1);
  mfma2<DT>(xv.z, av.z, c0, c1);
  mfma2<DT>(xv.w, av.w, c0, c1);
}

template <int DT>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  u.x = (uint32_t)Elem<DT>::from_float(f[0]) | ((uint32_t)Elem<DT>::from_float(f[1]) << 16);
  u.y = (uint32_t)Elem<DT>::from_float(f[2]) | ((uint32_t)Elem<DT>::from_float(f[3]) << 16);
  u.z = (uint32_t)Elem<DT>::from_float(f[4]) | ((uint32_t)Elem<DT>::from_float(f[5]) << 16);
  u.w = (uint32_t)Elem<DT>::from_float(f[6]) | ((uint32_t)Elem<DT>::from_float(f[7]) << 16);
  return u;
}

// ---- addresses ------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make the initialised barriers visible to the async proxy and to the cluster.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Default limit of a wait on data this kernel (or its cluster) is about to receive, and the limit
// of the waits that drain copies still in flight before a CTA that gave up exits.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 100000000ull;

// Non-blocking probes of a phase (mbarrier.test_wait): true once the phase with the given parity
// has completed. Unlike try_wait they never suspend the thread.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Limits below this are served by polling with test_wait and reading the clock at every poll:
// try_wait may suspend the thread for longer than such a limit.
constexpr uint64_t kShortLimitNs = 1000ull;

// Wait for the phase with the given parity to complete, for at most `limit_ns` nanoseconds.
// Returns false on timeout (the caller reports MLORA_STATUS_TIMEOUT and stops using the stage).
// The clock is read every 256 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (limit_ns < kShortLimitNs) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      if (mbar_test(bar, parity)) return true;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Same wait with cluster-scope acquire: for barriers completed by peers' st.async pushes.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (limit_ns < kShortLimitNs) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      if (mbar_test_cluster(bar, parity)) return true;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ---- programmatic dependent launch -------------------------------------------------------------

// Allow the next kernel in the stream to be scheduled now (it still waits for this grid to
// finish before griddepcontrol.wait returns in it).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One arrival on a shared-memory mbarrier (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Wait until every grid this one depends on has completed and its memory is visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- bulk copies (TMA, untiled) ---------------------------------------------------------------

// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global to this CTA's
// shared memory; completion is signalled to `bar` as a transaction count.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint for data read exactly once (adapter weights).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Prefetch `bytes` (multiple of 16, 16-byte aligned) of global memory into L2, asynchronously:
// nothing comes back to the SM and nothing is tracked. L2 is the point of coherence for the
// SMs, so a line prefetched before another kernel writes it is updated by that write.
__device__ __forceinline__ void prefetch_l2(const void *src_gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// 16-byte streaming load of data read once (no L1 allocation, evict-first in L2).
__device__ __forceinline__ uint4 ldg_stream(const void *p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// 16-byte load of data another kernel may have written (coherent path).
__device__ __forceinline__ uint4 ldg_u4(const void *p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// ---- clusters and distributed shared memory ------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Split cluster barrier: arrive (relaxed; the mbarrier-init fence already released the barriers)
// and, later, wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Store one float into a peer CTA's shared memory; the store completes as 4 transaction bytes
// on the peer's mbarrier (both addresses from mapa).
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote_addr), "f"(v),
               "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of the same variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ---- status ---------------------------------------------------------------------------------

__device__ __forceinline__ void report(int32_t *status, int32_t bits) {
  if (status && bits) atomicOr(status, bits);
}

}  // namespace mlora
