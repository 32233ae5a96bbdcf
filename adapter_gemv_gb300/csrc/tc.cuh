// tc.cuh -- Blackwell tensor-core helpers (sm_103a): tiled TMA loads, tcgen05 MMA with the
// accumulator in tensor memory (TMEM), and the shared-memory matrix descriptors they read.
//
// Operand layouts used here (16-bit elements, 128-byte swizzle):
//   K-major tile  : rows of 64 K-elements (128 B); 8 rows form a 1024-byte swizzle atom; the
//                   16-byte chunk c of row r sits at chunk position c ^ (r % 8). Stride between
//                   8-row groups (SBO) = 1024 B. One MMA consumes K = 16 (32 bytes of a row);
//                   the next K step starts 32 bytes further.
//   MN-major tile : rows of 64 MN-elements (128 B) per K index, same swizzle; SBO = 1024 B
//                   between 8-K-row groups, LBO = bytes between consecutive 64-wide MN atoms.
// A tiled TMA load with CU_TENSOR_MAP_SWIZZLE_128B and a 64-element inner box writes exactly
// these layouts.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace mlora {
namespace tc {

// ---- TMA -------------------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load of one box at (c0 = innermost coordinate, c1) into shared memory.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled store of one box from shared memory to (c0, c1); tracked as a bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, int c0, int c1, const void *src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(smem_u32(src))
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group has completed (its writes are performed).
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy (TMA, tensor cores).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- 16-byte asynchronous copies (global -> shared), for tiles gathered row by row ----------

// Copy 16 bytes (both addresses 16-byte aligned) into shared memory without registers; with
// src_bytes == 0 nothing is read and the 16 bytes are zero-filled.
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src_gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src_gmem),
               "r"(src_bytes)
               : "memory");
}

// One arrival on `bar` once every cp.async this thread issued so far has landed (the arrival is
// counted in the barrier's expected count: .noinc).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- TMEM --------------------------------------------------------------------------------------

// Whole warp: allocate `ncols` (power of two >= 32) TMEM columns; the address lands in *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- descriptors -------------------------------------------------------------------------------

// Shared-memory matrix descriptor (tcgen05 format): start, LBO and SBO in 16-byte units,
// version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void *p, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  const uint64_t addr = smem_u32(p);
  uint64_t d = (addr >> 4) & 0x3FFFull;
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= 2ull << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor for kind::f16 with an fp32 accumulator.
// ab_bf16: operands are bf16 (else fp16); a_mn / b_mn: operand stored MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_f16(bool ab_bf16, bool a_mn, bool b_mn, int M, int N) {
  return (1u << 4)                              // D format: f32
         | ((ab_bf16 ? 1u : 0u) << 7)           // A format
         | ((ab_bf16 ? 1u : 0u) << 10)          // B format
         | ((a_mn ? 1u : 0u) << 15)             // A major
         | ((b_mn ? 1u : 0u) << 16)             // B major
         | ((uint32_t)(N >> 3) << 17)           // N / 8
         | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// ---- MMA ---------------------------------------------------------------------------------------

// D[tmem] (+)= A[smem] x B[smem]; issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with the A operand in tensor memory (K-major: lane = row, two 16-bit elements per column).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrival when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---- registers -> TMEM ------------------------------------------------------------------------------

// 32 lanes x 4 consecutive 32-bit columns; the warp writes its own 32-lane quarter. Completion is
// awaited with tmem_st_wait().
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint4 &v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- TMEM -> registers ----------------------------------------------------------------------------

// 32 lanes x 16 consecutive 32-bit columns; the warp reads its own 32-lane quarter.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace tc
}  // namespace mlora
