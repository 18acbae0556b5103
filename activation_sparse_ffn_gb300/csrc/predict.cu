// Predictor kernels (PowerInfer §5.1 "Predictors" and the threshold note of
// its "Paper vs code" list): hid = ReLU(W1 . x + b1), s = W2 . hid + b2,
// slot i active iff s_i >= thres, emitted as a neuron bitmask with one warp
// ballot per 32 slots; plus the kernel that expands a bitmask into the
// ascending index list, the count and the group bitmask.
#include "common.cuh"
#include "internal.h"
#include "scan.cuh"

#include <algorithm>

namespace sffn {

namespace {

constexpr int kHidRows = 4;      // predictor rows per thread block (stage 1)
constexpr int kHidThreads = 256;
constexpr int kScoreThreads = 128;  // 4 warps split the hidden dimension (stage 2)
constexpr int kScorePreStages = 2;  // ring stages requested before the dependency wait (stage 2)
constexpr int kViewThreads = 1024;

// Stage 1: each block computes kHidRows rows of hid. Thread t owns the
// 16-byte chunks t, t+256, ... of every row, so the x values it needs are the
// same for all rows. The weights do not depend on the previous kernel, so all
// of a thread's weight loads are issued into registers before waiting for x;
// per-row partial sums are reduced across the block in a fixed order.
template <typename T, int CPT>
__global__ void __launch_bounds__(kHidThreads) k_pred_hidden(const T* __restrict__ W1, const float* __restrict__ b1,
                                                             const float* x, float* __restrict__ hid,
                                                             int h, int d) {
  constexpr int EPC = WType<T>::kPerChunk;
  const int r0 = blockIdx.x * kHidRows;
  const int nrows = min(kHidRows, h - r0);
  const T* base = W1 + (size_t)r0 * d;
  const int nch = d / EPC;
  uint4 w[kHidRows][CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * kHidThreads;
#pragma unroll
    for (int r = 0; r < kHidRows; ++r)
      if (r < nrows && c < nch) w[r][j] = ldg_stream(base + (size_t)r * d + (size_t)c * EPC);
  }
  pdl_launch_dependents();
  pdl_wait();

  float acc[kHidRows];
#pragma unroll
  for (int r = 0; r < kHidRows; ++r) acc[r] = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * kHidThreads;
    if (c < nch) {
      float xv[EPC];
#pragma unroll
      for (int e = 0; e < EPC; e += 4) {
        const float4 v = ld_dep4(x + (size_t)c * EPC + e);
        xv[e] = v.x; xv[e + 1] = v.y; xv[e + 2] = v.z; xv[e + 3] = v.w;
      }
#pragma unroll
      for (int r = 0; r < kHidRows; ++r)
        if (r < nrows) acc[r] += dot_chunk<T>(w[r][j], xv);
    }
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
    for (int w2 = 0; w2 < kHidThreads / 32; ++w2) s += red[w2][threadIdx.x];
    if (b1) s += b1[r0 + threadIdx.x];
    hid[r0 + threadIdx.x] = relu_nan(s);
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

// Stage 2: persistent blocks, each owning a contiguous range of mask words
// (32 consecutive slots = 32 contiguous W2 rows). The rows are streamed into a
// shared-memory ring one word per stage by bulk copies; the first stages are
// issued before waiting for hid. Warp w covers the w-th quarter of the hidden
// dimension for all 32 rows; lane sums are reduce-scattered so lane i holds
// row i; the four warp partials are added in a fixed order, the threshold is
// applied and one ballot gives the word.
template <typename T>
__global__ void __launch_bounds__(kScoreThreads, 1) k_pred_scores(const T* __restrict__ W2,
                                                                   const float* __restrict__ b2,
                                                                   const float* hid, float thres,
                                                                   uint32_t* __restrict__ nmask, int h, int nw,
                                                                   int stages, uint32_t* __restrict__ err) {
  constexpr int EPC = WType<T>::kPerChunk;
  const int nb = gridDim.x, b = blockIdx.x;
  const int w0 = (int)((long long)nw * b / nb), w1 = (int)((long long)nw * (b + 1) / nb);
  const int nloc = w1 - w0;
  const uint32_t row_bytes = (uint32_t)h * sizeof(T);
  const uint32_t word_bytes = 32u * row_bytes;
  extern __shared__ __align__(128) unsigned char smem[];
  float* s_hid = reinterpret_cast<float*>(smem + (size_t)stages * word_bytes);  // 16-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(s_hid + h);
  __shared__ float red[2][kScoreThreads / 32][32];
  __shared__ int s_issued;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_first();
  auto issue = [&](int k) {
    const int s = k % stages;
    mbar_arrive_expect_tx(&full[s], word_bytes);
    bulk_g2s(smem + (size_t)s * word_bytes, W2 + (size_t)(w0 + k) * 32 * h, word_bytes, &full[s], pol);
  };
  // The first kScorePreStages stages are requested before the wait, the rest
  // of the ring right after it: a larger burst before the wait delayed the
  // wait's return (measured on GB300, 70B-shaped layer: 45.0 us per layer with
  // the whole ring of 3 stages requested early, 44.4 with 1 or 2, 45.2 with 0).
  const int first = min(stages, nloc);
  const int pre = min(first, kScorePreStages);
  if (threadIdx.x == 0) {
    for (int k = 0; k < pre; ++k) issue(k);
    s_issued = first;
  }
  pdl_launch_dependents();
  pdl_wait();  // hid comes from the previous kernel
  if (threadIdx.x == 0)
    for (int k = pre; k < first; ++k) issue(k);
  for (int i = threadIdx.x * 4; i < h; i += kScoreThreads * 4)
    *reinterpret_cast<float4*>(s_hid + i) = ld_dep4(hid + i);
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = h / EPC;
  const int cpw = (nch + 3) / 4;
  const int c0 = warp * cpw, c1 = min(nch, c0 + cpw);
  int k = 0;
  bool aborted = false;
  for (; k < nloc; ++k) {
    const int s = k % stages;
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((k / stages) & 1));
    const unsigned char* sp = smem + (size_t)s * word_bytes;
    float acc[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) acc[r] = 0.f;
    for (int c = c0 + lane; c < c1; c += 32) {
      float hv[EPC];
#pragma unroll
      for (int e = 0; e < EPC; ++e) hv[e] = s_hid[c * EPC + e];
#pragma unroll
      for (int r = 0; r < 32; ++r)
        acc[r] += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + (size_t)r * row_bytes + (size_t)c * 16), hv);
    }
    transpose_reduce32(acc, lane);
    red[k & 1][warp][lane] = acc[0];
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (warp == 0) {
      float sc = red[k & 1][0][lane];
#pragma unroll
      for (int w2 = 1; w2 < kScoreThreads / 32; ++w2) sc += red[k & 1][w2][lane];
      if (b2) sc += b2[(size_t)(w0 + k) * 32 + lane];
      const uint32_t m = __ballot_sync(SFFN_FULL_MASK, sc >= thres);  // NaN compares false
      if (lane == 0) {
        nmask[w0 + k] = m;
        if (k + stages < nloc) {
          fence_proxy_async_smem();
          issue(k + stages);
          s_issued = k + stages + 1;
        }
      }
    }
  }
  if (aborted && threadIdx.x == 0) {
    set_device_error(err, SFFN_ERR_TIMEOUT);
    for (int q = k; q < s_issued; ++q) mbar_wait_bounded(&full[q % stages], (uint32_t)((q / stages) & 1));
  }
}

// Expands a neuron bitmask into the ascending index list, the count and the
// group bitmask (single block).
__global__ void __launch_bounds__(kViewThreads) k_mask_views(const uint32_t* nmask, int nw,
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

namespace {

int hid_cpt(const sffn_layer& L) {
  const int nch = L.desc.d * L.wbytes / 16;
  const int need = (nch + kHidThreads - 1) / kHidThreads;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
}

template <typename T>
cudaError_t launch_hidden_t(const sffn_layer& L, const float* x, float* hid, cudaStream_t st) {
  const int h = L.desc.h, d = L.desc.d;
  const dim3 grid((h + kHidRows - 1) / kHidRows), block(kHidThreads);
  const T* W1 = static_cast<const T*>(L.W1);
  const float* b1 = L.has_b1 ? L.b1 : nullptr;
  switch (hid_cpt(L)) {
    case 1: return launch_ex(k_pred_hidden<T, 1>, grid, block, 0, st, true, 1, W1, b1, x, hid, h, d);
    case 2: return launch_ex(k_pred_hidden<T, 2>, grid, block, 0, st, true, 1, W1, b1, x, hid, h, d);
    case 4: return launch_ex(k_pred_hidden<T, 4>, grid, block, 0, st, true, 1, W1, b1, x, hid, h, d);
    default: return launch_ex(k_pred_hidden<T, 8>, grid, block, 0, st, true, 1, W1, b1, x, hid, h, d);
  }
}

template <typename T>
cudaError_t launch_scores_t(const sffn_layer& L, const float* hid, float thres, uint32_t* nmask, cudaStream_t st) {
  const dim3 grid(std::min(L.nwords, L.score_grid > 0 ? L.score_grid : L.num_sms)), block(kScoreThreads);
  const float* b2 = L.has_b2 ? L.b2 : nullptr;
  return launch_ex(k_pred_scores<T>, grid, block, score_smem(L), st, true, 1, static_cast<const T*>(L.W2), b2, hid,
                   thres, nmask, L.desc.h, L.nwords, L.score_stages, L.err);
}

}  // namespace

int score_stages_for(const sffn_layer& L) {
  const size_t word = (size_t)32 * L.desc.h * L.wbytes;
  return (int)std::min<size_t>(6, std::max<size_t>(2, kScoreSmemBudget / word));
}

size_t score_smem(const sffn_layer& L) {
  return (size_t)L.score_stages * 32 * L.desc.h * L.wbytes + (size_t)L.score_stages * 8 + (size_t)L.desc.h * 4;
}

template <typename K>
cudaError_t carveout_max(K* kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

template <typename T>
cudaError_t configure_predict_t(int sm) {
  // every hot kernel asks for the largest shared-memory carveout, so that
  // consecutive kernels of a decode step need no L1/shared reconfiguration
  cudaError_t e = set_dynamic_smem_max(k_pred_scores<T>, sm);
  if (e == cudaSuccess) e = carveout_max(k_pred_scores<T>);
  if (e == cudaSuccess) e = carveout_max(k_pred_hidden<T, 1>);
  if (e == cudaSuccess) e = carveout_max(k_pred_hidden<T, 2>);
  if (e == cudaSuccess) e = carveout_max(k_pred_hidden<T, 4>);
  if (e == cudaSuccess) e = carveout_max(k_pred_hidden<T, 8>);
  if (e == cudaSuccess) e = carveout_max(k_mask_views);
  return e;
}

// The limit is the device maximum (shared by all layers; see configure_kernels).
cudaError_t configure_predict_kernels(const sffn_layer& L) {
  if (score_smem(L) + 2048 > (size_t)L.smem_optin) return cudaErrorInvalidConfiguration;
  const int sm = L.smem_optin;
  switch (L.desc.wdtype) {
    case SFFN_F32: return configure_predict_t<float>(sm);
    case SFFN_F16: return configure_predict_t<__half>(sm);
    default: return configure_predict_t<__nv_bfloat16>(sm);
  }
}

cudaError_t launch_pred_hidden(const sffn_layer& L, const float* x, float* hid, cudaStream_t st) {
  switch (L.desc.wdtype) {
    case SFFN_F32: return launch_hidden_t<float>(L, x, hid, st);
    case SFFN_F16: return launch_hidden_t<__half>(L, x, hid, st);
    default: return launch_hidden_t<__nv_bfloat16>(L, x, hid, st);
  }
}

cudaError_t launch_pred_scores(const sffn_layer& L, const float* hid, float thres, uint32_t* nmask,
                               cudaStream_t st) {
  switch (L.desc.wdtype) {
    case SFFN_F32: return launch_scores_t<float>(L, hid, thres, nmask, st);
    case SFFN_F16: return launch_scores_t<__half>(L, hid, thres, nmask, st);
    default: return launch_scores_t<__nv_bfloat16>(L, hid, thres, nmask, st);
  }
}

cudaError_t launch_mask_views(const sffn_layer& L, const uint32_t* nmask, int32_t* idx, int32_t* count,
                              uint32_t* gmask, cudaStream_t st) {
  const size_t smem = (size_t)L.nwords * 8;
  return launch_ex(k_mask_views, dim3(1), dim3(kViewThreads), smem, st, true, 1, nmask, L.nwords, L.n_groups,
                   L.desc.group_size, L.gwords, idx, count, gmask);
}

}  // namespace sffn
