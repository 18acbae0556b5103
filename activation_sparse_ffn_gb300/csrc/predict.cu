// Predictor kernels (PowerInfer §5.1 "Predictors" and the threshold note of
// its "Paper vs code" list): hid = ReLU(W1 . x + b1), s = W2 . hid + b2,
// slot i active iff s_i >= thres, emitted as a neuron bitmask with one warp
// ballot per 32 slots; plus the kernel that expands a bitmask into the
// ascending index list, the count and the group bitmask.
#include "common.cuh"
#include "internal.h"
#include "scan.cuh"

namespace sffn {

namespace {

constexpr int kHidRows = 8;      // predictor rows per thread block (stage 1)
constexpr int kHidThreads = 256;
constexpr int kScoreThreads = 128;  // 4 warps per 32-row mask word (stage 2)
constexpr int kViewThreads = 1024;

// Stage 1: each block computes kHidRows rows of hid. Thread t owns the
// 16-byte chunks t, t+256, ... of every row, so the x values it needs are
// the same for all rows; per-row partial sums are reduced across the block
// in a fixed order.
template <typename T>
__global__ void __launch_bounds__(kHidThreads) k_pred_hidden(const T* __restrict__ W1, const float* __restrict__ b1,
                                                             const float* __restrict__ x, float* __restrict__ hid,
                                                             int h, int d) {
  constexpr int EPC = WType<T>::kPerChunk;
  const int r0 = blockIdx.x * kHidRows;
  const int nrows = min(kHidRows, h - r0);
  const T* base = W1 + (size_t)r0 * d;
  // The weights do not depend on the previous kernel: start pulling this
  // block's rows into L2 before waiting for x.
  if (threadIdx.x == 0) prefetch_l2_bulk(base, (uint32_t)((size_t)nrows * d * sizeof(T)));
  pdl_launch_dependents();
  pdl_wait();

  const int nch = d / EPC;
  float acc[kHidRows];
#pragma unroll
  for (int r = 0; r < kHidRows; ++r) acc[r] = 0.f;
  for (int c = threadIdx.x; c < nch; c += kHidThreads) {
    float xv[EPC];
#pragma unroll
    for (int e = 0; e < EPC; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(x + c * EPC + e);
      xv[e] = v.x; xv[e + 1] = v.y; xv[e + 2] = v.z; xv[e + 3] = v.w;
    }
    uint4 w[kHidRows];
#pragma unroll
    for (int r = 0; r < kHidRows; ++r)
      if (r < nrows) w[r] = ldg_stream(base + (size_t)r * d + (size_t)c * EPC);
#pragma unroll
    for (int r = 0; r < kHidRows; ++r)
      if (r < nrows) acc[r] += dot_chunk<T>(w[r], xv);
  }
  __shared__ float red[kHidThreads / 32][kHidRows];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < kHidRows; ++r) {
    const float v = warp_sum(acc[r]);
    if (lane == 0) red[warp][r] = v;
  }
  __syncthreads();
  if (threadIdx.x < nrows) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kHidThreads / 32; ++w) s += red[w][threadIdx.x];
    if (b1) s += b1[r0 + threadIdx.x];
    hid[r0 + threadIdx.x] = fmaxf(s, 0.f);
  }
}

// Butterfly reduce-scatter of 32 per-lane partial sums: afterwards lane i
// holds the warp-wide sum of partial i in v[0] (31 shuffles).
__device__ __forceinline__ void transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < off; ++j) {
      const float send = upper ? v[j] : v[j + off];
      const float keep = upper ? v[j + off] : v[j];
      v[j] = keep + __shfl_xor_sync(SFFN_FULL_MASK, send, off);
    }
  }
}

// Stage 2: one block per mask word (32 consecutive slots). Warp w covers the
// w-th quarter of the hidden dimension for all 32 rows; lane sums are
// reduce-scattered so lane i holds row i; the four warp partials are added in
// a fixed order, the threshold is applied and one ballot gives the word.
template <typename T>
__global__ void __launch_bounds__(kScoreThreads, 6) k_pred_scores(const T* __restrict__ W2,
                                                                   const float* __restrict__ b2,
                                                                   const float* __restrict__ hid, float thres,
                                                                   uint32_t* __restrict__ nmask, int h) {
  constexpr int EPC = WType<T>::kPerChunk;
  const int word = blockIdx.x;
  const T* base = W2 + (size_t)word * 32 * h;
  if (threadIdx.x == 0) prefetch_l2_bulk(base, (uint32_t)((size_t)32 * h * sizeof(T)));
  pdl_launch_dependents();
  pdl_wait();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = h / EPC;
  const int cpw = (nch + 3) / 4;
  const int c0 = warp * cpw, c1 = min(nch, c0 + cpw);
  float acc[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) acc[r] = 0.f;
  for (int c = c0 + lane; c < c1; c += 32) {
    float hv[EPC];
#pragma unroll
    for (int e = 0; e < EPC; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(hid + c * EPC + e);
      hv[e] = v.x; hv[e + 1] = v.y; hv[e + 2] = v.z; hv[e + 3] = v.w;
    }
#pragma unroll
    for (int r0 = 0; r0 < 32; r0 += 8) {
      uint4 w[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) w[r] = ldg_stream(base + (size_t)(r0 + r) * h + (size_t)c * EPC);
#pragma unroll
      for (int r = 0; r < 8; ++r) acc[r0 + r] += dot_chunk<T>(w[r], hv);
    }
  }
  transpose_reduce32(acc, lane);
  __shared__ float red[kScoreThreads / 32][32];
  red[warp][lane] = acc[0];
  __syncthreads();
  if (warp == 0) {
    float s = red[0][lane];
#pragma unroll
    for (int w = 1; w < kScoreThreads / 32; ++w) s += red[w][lane];
    if (b2) s += b2[word * 32 + lane];
    const uint32_t m = __ballot_sync(SFFN_FULL_MASK, s >= thres);  // NaN compares false
    if (lane == 0) nmask[word] = m;
  }
}

// Expands a neuron bitmask into the ascending index list, the count and the
// group bitmask (single block).
__global__ void __launch_bounds__(kViewThreads) k_mask_views(const uint32_t* __restrict__ nmask, int nw,
                                                             int n_groups, int G, int gwords,
                                                             int32_t* __restrict__ idx, int32_t* __restrict__ count,
                                                             uint32_t* __restrict__ gmask) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* s_words = reinterpret_cast<uint32_t*>(smem);
  int* s_off = reinterpret_cast<int*>(s_words + nw);
  __shared__ int s_tmp[kViewThreads / 32];
  const int total = scan_mask_words<kViewThreads>(nmask, nw, s_words, s_off, s_tmp);
  if (idx) extract_slice<kViewThreads>(s_words, s_off, nw, 0, total, idx);
  if (count && threadIdx.x == 0) *count = total;
  if (gmask) write_group_mask<kViewThreads>(s_words, n_groups, G, gwords, gmask);
}

}  // namespace

cudaError_t launch_pred_hidden(const sffn_layer& L, const float* x, float* hid, cudaStream_t st) {
  const int h = L.desc.h, d = L.desc.d;
  dim3 grid((h + kHidRows - 1) / kHidRows);
  const float* b1 = L.has_b1 ? L.b1 : nullptr;
  switch (L.desc.wdtype) {
    case SFFN_F32:
      return launch_ex(k_pred_hidden<float>, grid, dim3(kHidThreads), 0, st, true, 1,
                       static_cast<const float*>(L.W1), b1, x, hid, h, d);
    case SFFN_F16:
      return launch_ex(k_pred_hidden<__half>, grid, dim3(kHidThreads), 0, st, true, 1,
                       static_cast<const __half*>(L.W1), b1, x, hid, h, d);
    default:
      return launch_ex(k_pred_hidden<__nv_bfloat16>, grid, dim3(kHidThreads), 0, st, true, 1,
                       static_cast<const __nv_bfloat16*>(L.W1), b1, x, hid, h, d);
  }
}

cudaError_t launch_pred_scores(const sffn_layer& L, const float* hid, float thres, uint32_t* nmask,
                               cudaStream_t st) {
  const int h = L.desc.h;
  dim3 grid(L.nwords);
  const float* b2 = L.has_b2 ? L.b2 : nullptr;
  switch (L.desc.wdtype) {
    case SFFN_F32:
      return launch_ex(k_pred_scores<float>, grid, dim3(kScoreThreads), 0, st, true, 1,
                       static_cast<const float*>(L.W2), b2, hid, thres, nmask, h);
    case SFFN_F16:
      return launch_ex(k_pred_scores<__half>, grid, dim3(kScoreThreads), 0, st, true, 1,
                       static_cast<const __half*>(L.W2), b2, hid, thres, nmask, h);
    default:
      return launch_ex(k_pred_scores<__nv_bfloat16>, grid, dim3(kScoreThreads), 0, st, true, 1,
                       static_cast<const __nv_bfloat16*>(L.W2), b2, hid, thres, nmask, h);
  }
}

cudaError_t launch_mask_views(const sffn_layer& L, const uint32_t* nmask, int32_t* idx, int32_t* count,
                              uint32_t* gmask, cudaStream_t st) {
  const size_t smem = (size_t)L.nwords * 8;
  return launch_ex(k_mask_views, dim3(1), dim3(kViewThreads), smem, st, true, 1, nmask, L.nwords, L.n_groups,
                   L.desc.group_size, L.gwords, idx, count, gmask);
}

}  // namespace sffn
