// Fifth-generation tensor core (tcgen05) helpers for sm_103a: tensor-memory
// allocation, shared-memory matrix descriptors for 128-byte-swizzled
// operands, the kind::f16 MMA, commit to an mbarrier, and tensor-memory loads.
//
// Operand layouts (16-bit elements, 128-byte swizzle; every tile base is
// 1024-byte aligned):
//   K-major tile, R rows x 64 K: row r at r*128 bytes, its 16-byte chunk j
//     (elements 8j..8j+7) at chunk position j ^ (r & 7). Descriptor: LBO 16,
//     SBO 1024 (eight-row groups); the K step of 16 advances the start address
//     by 32 bytes.
//   MN-major tile, 128 M x 64 K: eight-K-row atoms of 64 M elements (128-byte
//     rows); atom (k/8, m/64) at (k/8)*2048 + (m/64)*1024; within an atom K row
//     kr at kr*128 and the 16-byte chunk of M elements c at (c ^ kr)*16.
//     Descriptor: LBO 1024 (stride between M-adjacent atoms), SBO 2048 (between
//     K-adjacent atoms); the K step of 16 advances the start by 4096 bytes.
#pragma once

#include "common.cuh"

namespace sffn {
namespace tc {

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16
// (bf16 = true) or both fp16, B K-major, A K-major or MN-major, M = 128.
__host__ __device__ constexpr uint32_t instr_desc(bool bf16, bool a_mn_major, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                    bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// The mbarrier receives one arrival once every previously issued MMA of this
// thread has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Executed by one full warp.
__device__ __forceinline__ void alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Executed by the warp that allocated.
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 16 columns of 32-bit values: thread l of the warp gets lane
// (row) base_lane + l, columns col..col+15.
__device__ __forceinline__ void ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16-byte asynchronous copy global -> shared through L2 (not L1), read under
// the given L2 eviction policy.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src),
               "l"(policy)
               : "memory");
}

// One arrival on the mbarrier once all of this thread's earlier cp.async
// copies have landed (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Two-dimensional tiled TMA load of the box at element coordinates (x, y) of
// the tensor map into shared memory at dst (1024-byte aligned for the
// 128-byte swizzle); completion is signalled on `bar` as transaction bytes.
// x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Byte offset of 16-byte chunk j (0..7) of row r in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t kmajor_off(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) * 16)); }

// Byte offset of the 16-byte chunk holding M elements [8c, 8c+8) of K row k in
// an MN-major 128 x 64 tile (c in 0..15).
__device__ __forceinline__ uint32_t mnmajor_off(int k, int c) {
  const int ka = k >> 3, kr = k & 7, ma = c >> 3, mc = c & 7;
  return (uint32_t)(ka * 2048 + ma * 1024 + kr * 128 + ((mc ^ kr) * 16));
}

}  // namespace tc
}  // namespace sffn
