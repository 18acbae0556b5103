// Temporal activation momentum (KAIROX review page, 核心方法 item 4) and the
// Adaptive Neuron Balancer step (item 5), one thread block per layer.
//
// Momentum update, float32 with one rounding per operation (no fused
// multiply-add): om = 1 - lambda, tau = om + eps, s = lambda * s, then
// s = s + om for an active group. Candidates are groups with s > tau; the
// first capacity_k candidates ranked by (s descending, group ascending) stay
// resident, found by a bitonic sort of packed keys (float bits of s, then the
// complement of the group id) over at most 1024 groups in shared memory. The
// load / evict / changed sets are the fused AND-NOT and XOR of the bitsets
// (item 6).
#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int kTamThreads = 1024;

__global__ void __launch_bounds__(kTamThreads)
    k_tam_update(float* scores, const float* lambdas, uint32_t* resident,
                 int n_groups, int gwords, const uint32_t* gmask, int gstride, int layer0,
                 float lambda_arg, float eps, int K, tam_outputs out) {
  pdl_launch_dependents();
  pdl_wait();
  const int l = blockIdx.x;
  const int layer = layer0 + l;
  const int g = threadIdx.x;
  const int lane = g & 31, warp = g >> 5;
  __shared__ unsigned long long keys[kTamThreads];
  __shared__ uint32_t s_cand[32], s_res[32];

  const float lam = lambda_arg >= 0.f ? lambda_arg : ld_dep(lambdas + layer);
  const float om = __fsub_rn(1.0f, lam);
  const float tau = __fadd_rn(om, eps);
  float s = 0.f;
  bool c = false;
  if (g < n_groups) {
    float* sp = scores + (size_t)layer * n_groups + g;
    const bool active = (ld_dep(gmask + (size_t)l * gstride + (g >> 5)) >> (g & 31)) & 1u;
    s = __fmul_rn(lam, ld_dep(sp));
    s = __fadd_rn(s, active ? om : 0.0f);
    *sp = s;
    c = s > tau;
  }
  const uint32_t cw = __ballot_sync(SFFN_FULL_MASK, c);
  if (lane == 0) s_cand[warp] = cw;
  if (g < 32) s_res[g] = 0u;
  unsigned long long key =
      c ? ((unsigned long long)__float_as_uint(s) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)g) : 0ull;
  const int nc = __syncthreads_count(c);
  // Bitonic sort, descending. Partner distances j >= 32 exchange through
  // shared memory (one barrier per step); j < 32 exchange with warp shuffles.
  // In a block of size k that sorts descending ((g & k) == 0) the lower index
  // of each pair keeps the larger key; in an ascending block, the smaller.
  for (int k = 2; k <= kTamThreads; k <<= 1) {
    const bool desc = (g & k) == 0;
    int j = k >> 1;
    if (j >= 32) {
      keys[g] = key;
      __syncthreads();
      for (; j >= 32; j >>= 1) {
        const int p = g ^ j;
        if (p > g) {
          const unsigned long long a = keys[g], b = keys[p];
          if (desc ? (a < b) : (a > b)) {
            keys[g] = b;
            keys[p] = a;
          }
        }
        __syncthreads();
      }
      key = keys[g];
      __syncthreads();
    }
    for (; j > 0; j >>= 1) {
      const unsigned long long other = __shfl_xor_sync(SFFN_FULL_MASK, key, j);
      const bool lower = (g & j) == 0;
      const unsigned long long hi = key > other ? key : other, lo2 = key > other ? other : key;
      key = (lower == desc) ? hi : lo2;
    }
  }
  keys[g] = key;
  __syncthreads();
  const int nres = min(K, nc);
  int gid = -1;
  if (g < nres) {
    gid = (int)(0xffffffffu - (uint32_t)(keys[g] & 0xffffffffull));
    atomicOr(&s_res[gid >> 5], 1u << (gid & 31));
  }
  if (out.topk && g < K) out.topk[(size_t)l * K + g] = gid;
  __syncthreads();
  if (g < gwords) {
    uint32_t* rp = resident + (size_t)layer * gwords + g;
    const uint32_t prev = ld_dep(rp), res = s_res[g];
    const size_t o = (size_t)l * gwords + g;
    if (out.cand) out.cand[o] = s_cand[g];
    if (out.resident) out.resident[o] = res;
    if (out.load) out.load[o] = res & ~prev;
    if (out.evict) out.evict[o] = prev & ~res;
    if (out.changed) out.changed[o] = res ^ prev;
    *rp = res;
  }
  if (g == 0) {
    if (out.n_cand) out.n_cand[l] = nc;
    if (out.n_res) out.n_res[l] = nres;
  }
}

__global__ void k_tam_adapt(float* lambdas, int layer0, int n, const uint8_t* stall,
                            float alpha, float lo, float hi) {
  pdl_launch_dependents();
  pdl_wait();
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  if (l < n) {
    const float v = __fadd_rn(ld_dep(lambdas + layer0 + l), __ldcg(stall + l) ? alpha : -alpha);
    lambdas[layer0 + l] = fminf(hi, fmaxf(lo, v));
  }
}

// One block waits on a barrier that nothing completes; the bounded wait runs
// out and records SFFN_ERR_TIMEOUT. Exercises the timeout path without a fault.
__global__ void k_selftest_timeout(uint32_t* __restrict__ err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
  if (__syncthreads_or(!ok) && threadIdx.x == 0) set_device_error(err, SFFN_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_tam_update(tam_state& S, int layer0, int n_layers, const uint32_t* gmask, int gstride,
                              float lambda, float eps, int K, const tam_outputs& out, cudaStream_t st) {
  return launch_ex(k_tam_update, dim3(n_layers), dim3(kTamThreads), 0, st, true, 1, S.scores,
                   static_cast<const float*>(S.lambdas), S.resident, S.n_groups, S.gwords, gmask, gstride, layer0,
                   lambda, eps, K, out);
}

cudaError_t launch_tam_adapt(tam_state& S, int layer0, int n_layers, const uint8_t* stall, float alpha, float lo,
                             float hi, cudaStream_t st) {
  return launch_ex(k_tam_adapt, dim3((n_layers + 127) / 128), dim3(128), 0, st, true, 1, S.lambdas, layer0,
                   n_layers, stall, alpha, lo, hi);
}

cudaError_t launch_selftest_timeout(uint32_t* err, int limit_us, cudaStream_t st) {
  return launch_ex(k_selftest_timeout, dim3(1), dim3(32), 0, st, false, 1, err,
                   (unsigned long long)limit_us * 1000ull);
}

}  // namespace sffn
