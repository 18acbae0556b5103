// Device-side helpers shared by the sffn kernels: inline PTX for shared-memory
// barriers (mbarrier), one-dimensional bulk copies global -> shared (the
// Blackwell TMA engine), L2 bulk prefetch, programmatic dependent launch, and
// weight-type conversions. sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sffn.h"

#define SFFN_FULL_MASK 0xffffffffu

namespace sffn {

// ----------------------------------------------------------------- errors

// Device error word: the first error code written wins.
__device__ __forceinline__ void set_device_error(uint32_t* err, uint32_t code) {
  if (err) atomicCAS(err, 0u, code);
}

// ----------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy accesses of shared memory before later
// async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Default bound of every device-side wait: one second.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Wait for the barrier phase with the given parity; gives up after limit_ns
// and returns false (the caller records SFFN_ERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Lines read under this policy are the last to leave L2.
__device__ __forceinline__ uint64_t l2_policy_keep() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// One-dimensional bulk copy global -> this CTA's shared memory; completion is
// signalled on `bar` as transaction bytes. dst, src and bytes must be
// multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Ask L2 to fetch [src, src + bytes) (bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Raise a kernel's dynamic shared-memory limit to what the device allows next
// to the kernel's own static shared memory. Kernel attributes are shared by
// every layer in the process, so the limit is set to the device maximum
// rather than to one layer's need.
template <typename K>
inline cudaError_t set_dynamic_smem_max(K* kern, int optin) {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, kern);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)a.sharedSizeBytes);
}

// Programmatic dependent launch: wait until the preceding kernel in the stream
// has completed and its writes are visible (a no-op without the launch
// attribute); allow the next kernel to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Loads of data written by an earlier kernel of the same stream, in
// particular by the programmatic-launch predecessor that this kernel waits for
// with griddepcontrol.wait. Such data is not read-only for this kernel's
// lifetime (the kernel starts before its predecessor finishes), so it must
// never go through the non-coherent read-only path (ld.global.nc, which
// `const __restrict__` pointers invite) or a possibly stale L1 line: these
// loads read from L2, the point of coherence, and are issued only after the
// wait.
__device__ __forceinline__ float ld_dep(const float* p) { return __ldcg(p); }
__device__ __forceinline__ int ld_dep(const int* p) { return __ldcg(p); }
__device__ __forceinline__ uint32_t ld_dep(const uint32_t* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ld_dep4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// 16-byte streaming load that does not allocate in L1 (immutable weights only).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ----------------------------------------------------------------- weight types

template <typename T>
struct WType;

template <>
struct WType<float> {
  static constexpr int kPerChunk = 4;  // elements per 16-byte chunk
  __device__ __forceinline__ static void unpack(const uint4& v, float* o) {
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
  }
};

template <>
struct WType<__half> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 p = *reinterpret_cast<const __half2*>(&w[i]);
      float2 f = __half22float2(p);
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
};

template <>
struct WType<__nv_bfloat16> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // a bfloat16 is the upper half of a float32
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// 8-bit codes of quantized FFN rows (the row's scale is applied by the caller).
template <>
struct WType<int8_t> {
  static constexpr int kPerChunk = 16;
  // Exact conversion with full-rate instructions only (an int-to-float
  // conversion issues at a fraction of the FMA rate): flipping the sign bit
  // turns code b into the unsigned byte u = b + 128; placing u in the low
  // byte of the bit pattern 0x4B000000 gives the float 2^23 + u exactly; one
  // subtraction of 2^23 + 128 leaves b.
  __device__ __forceinline__ static void unpack(const uint4& v, float* o) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    constexpr float kBias = 8388608.f + 128.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[4 * i + j] = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7440u | j)) - kBias;
    }
  }
  // The same as pairs (elements 2p, 2p+1), the bias removed two at a time.
  __device__ __forceinline__ static void unpack2(const uint4& v, float2* o) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    const float2 nb = make_float2(-(8388608.f + 128.f), -(8388608.f + 128.f));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < 4; j += 2)
        o[2 * i + j / 2] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7440u | j)),
                                                  __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7441u | j))),
                                      nb);
    }
  }
};

// Two signed 4-bit codes in one byte: element 2i in the low half of byte i,
// element 2i + 1 in the high half (the row's scale is applied by the caller).
struct q4x2_t {
  uint8_t v;
};

template <>
struct WType<q4x2_t> {
  static constexpr int kPerChunk = 32;
  // The 8-bit trick on half-bytes: masking out the low (or high, shifted
  // down) halves of a word leaves four 4-bit two's-complement codes c, one
  // per byte; flipping bit 3 turns each into c + 8 in [0, 15]; that byte in
  // the low byte of 0x4B000000 is the float 2^23 + c + 8, exact; subtracting
  // 2^23 + 8 leaves c.
  __device__ __forceinline__ static void unpack(const uint4& v, float* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    constexpr float kBias = 8388608.f + 8.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (w[i] & 0x0F0F0F0Fu) ^ 0x08080808u, hi = ((w[i] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o[8 * i + 2 * j] = __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u | j)) - kBias;
        o[8 * i + 2 * j + 1] = __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u | j)) - kBias;
      }
    }
  }
  // The same as pairs (elements 2p, 2p+1): a pair is the two halves of one byte.
  __device__ __forceinline__ static void unpack2(const uint4& v, float2* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float2 nb = make_float2(-(8388608.f + 8.f), -(8388608.f + 8.f));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (w[i] & 0x0F0F0F0Fu) ^ 0x08080808u, hi = ((w[i] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[4 * i + j] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u | j)),
                                              __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u | j))),
                                  nb);
    }
  }
};

// Dot product of one 16-byte weight chunk with kPerChunk fp32 values.
template <typename T>
__device__ __forceinline__ float dot_chunk(const uint4& w, const float* x) {
  float v[WType<T>::kPerChunk];
  WType<T>::unpack(w, v);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < WType<T>::kPerChunk; ++i) s = fmaf(v[i], x[i], s);
  return s;
}

// Dot product of one 16-byte chunk of codes with kPerChunk fp32 values held
// as pairs, in packed fp32 arithmetic with two independent accumulators.
template <typename T>
__device__ __forceinline__ float dot_chunk_pairs(const uint4& w, const float2* x) {
  constexpr int NP = WType<T>::kPerChunk / 2;
  float2 v[NP];
  WType<T>::unpack2(w, v);
  float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
  for (int p = 0; p < NP; p += 2) {
    a = __ffma2_rn(v[p], x[p], a);
    b = __ffma2_rn(v[p + 1], x[p + 1], b);
  }
  return (a.x + a.y) + (b.x + b.y);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(SFFN_FULL_MASK, v, o);
  return v;
}

// ReLU that propagates NaN (fmaxf would turn NaN into 0).
__device__ __forceinline__ float relu_nan(float v) { return v < 0.f ? 0.f : v; }

// Activation of one neuron from its up value u and gate value g.
template <int ACT>
__device__ __forceinline__ float neuron_act(float u, float g) {
  if (ACT == SFFN_ACT_RELU) return relu_nan(u);
  if (ACT == SFFN_ACT_RELU2) {
    const float r = relu_nan(u);
    return r * r;
  }
  if (ACT == SFFN_ACT_REGLU) return relu_nan(g) * u;
  return g / (1.f + expf(-g)) * u;  // SiLU(g) * u
}

}  // namespace sffn
