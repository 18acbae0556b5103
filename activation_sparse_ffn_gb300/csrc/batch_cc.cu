// CUDA-core arm of the batched decode step for 2..4 tokens (the tensor-core
// arm is batch.cu). Every weight row the batch needs is read once for all of
// its tokens, the way the B = 1 kernels read it for one (PowerInfer §5.1
// predictor, §5.3-§5.4 neuron-aware operators; KAIROX 问题与动机: the batch
// reads the union of its tokens' active rows):
//   k_cc_hidden  hid[b] = ReLU(W1 . x_b + b1): W1 rows in registers, the
//                tokens' x read per 16-byte chunk;
//   k_cc_scores  s[b] = W2 . hid[b] + b2, one ballot per token and word, and
//                the union word (OR over the tokens);
//   k_cc_ffn     the union slice of every block: up/gate rows through the
//                TMA ring, NB dot products per row (x of every token in
//                registers), h of token b is zero unless the neuron is in
//                token b's own mask, then NB partial sums of y per block;
//   k_cc_reduce  y[b] and x[b] + y[b] from the partials in a fixed order.
// fp32 FFMA arithmetic throughout. Each token's result is that of a B = 1
// call with the same per-token mask up to fp32 summation order: the union
// only decides which rows are read.
#include "common.cuh"
#include "internal.h"
#include "scan.cuh"

#include <algorithm>

namespace sffn {

namespace {

constexpr int kCcHidRows = 4;
constexpr int kCcHidThreads = 256;
constexpr int kCcScoreThreads = 128;
constexpr int kCcScorePreStages = 2;                // W2 ring stages requested before the dependency wait
constexpr int kCcWarps = 8;                       // FFN consumer warps
constexpr int kCcConsumers = kCcWarps * 32;
constexpr int kCcThreads = kCcConsumers + 32;     // + producer warp
constexpr int kCcReduceThreads = 256;
constexpr int kCcReduceCols = 32;
constexpr int kCcReduceGroups = kCcReduceThreads / (kCcReduceCols / 4);
constexpr int kCcCpt = 4;                         // 16-byte chunks per consumer thread and row (d <= 8192)
constexpr uint32_t kCcStageBytes = 32768;         // FFN ring stage

__device__ __forceinline__ void cc_consumer_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCcConsumers) : "memory");
}

template <typename T, int CPT, int NB>
__global__ void __launch_bounds__(kCcHidThreads) k_cc_hidden(const T* __restrict__ W1, const float* __restrict__ b1,
                                                             const float* x, int B, float* __restrict__ hid, int h,
                                                             int d) {
  constexpr int EPC = WType<T>::kPerChunk;
  const int r0 = blockIdx.x * kCcHidRows;
  const int nrows = min(kCcHidRows, h - r0);
  const int nch = d / EPC;
  uint4 w[kCcHidRows][CPT];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * kCcHidThreads;
#pragma unroll
    for (int r = 0; r < kCcHidRows; ++r)
      if (r < nrows && c < nch) w[r][j] = ldg_stream(W1 + (size_t)(r0 + r) * d + (size_t)c * EPC);
  }
  pdl_launch_dependents();
  pdl_wait();
  float acc[kCcHidRows][NB];
#pragma unroll
  for (int r = 0; r < kCcHidRows; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * kCcHidThreads;
    if (c < nch) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float xv[EPC];
#pragma unroll
        for (int e = 0; e < EPC; e += 4) {
          const float4 v = b < B ? ld_dep4(x + (size_t)b * d + (size_t)c * EPC + e) : make_float4(0.f, 0.f, 0.f, 0.f);
          xv[e] = v.x; xv[e + 1] = v.y; xv[e + 2] = v.z; xv[e + 3] = v.w;
        }
#pragma unroll
        for (int r = 0; r < kCcHidRows; ++r)
          if (r < nrows) acc[r][b] += dot_chunk<T>(w[r][j], xv);
      }
    }
  }
  __shared__ float red[kCcHidThreads / 32][kCcHidRows][NB];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < kCcHidRows; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float v = warp_sum(acc[r][b]);
      if (lane == 0) red[warp][r][b] = v;
    }
  __syncthreads();
  if (threadIdx.x < nrows * NB && (int)(threadIdx.x % NB) < B) {
    const int r = threadIdx.x / NB, b = threadIdx.x % NB;
    float s = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kCcHidThreads / 32; ++w2) s += red[w2][r][b];
    if (b1) s += b1[r0 + r];
    hid[(size_t)b * h + r0 + r] = relu_nan(s);
  }
}

// Butterfly reduce-scatter: lane i ends with the warp-wide sum of v[i].
__device__ __forceinline__ void cc_transpose_reduce32(float (&v)[32], int lane) {
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

// Persistent blocks over contiguous ranges of mask words, W2 rows of one word
// per ring stage; every token's 32 sums of a stage are formed in one pass over
// the stage (each weight chunk read from shared memory once for all tokens).
template <typename T, int NB>
__global__ void __launch_bounds__(kCcScoreThreads, 1)
    k_cc_scores(const T* __restrict__ W2, const float* __restrict__ b2, const float* hid, int B, float thres,
                uint32_t* __restrict__ nmask, uint32_t* __restrict__ unmask, int h, int nw, int stages,
                uint32_t* __restrict__ err) {
  constexpr int EPC = WType<T>::kPerChunk;
  const int nb = gridDim.x, blk = blockIdx.x;
  const int w0 = (int)((long long)nw * blk / nb), w1 = (int)((long long)nw * (blk + 1) / nb);
  const int nloc = w1 - w0;
  const uint32_t row_bytes = (uint32_t)h * sizeof(T);
  const uint32_t word_bytes = 32u * row_bytes;
  extern __shared__ __align__(128) unsigned char smem[];
  float* s_hid = reinterpret_cast<float*>(smem + (size_t)stages * word_bytes);  // [NB][h]
  uint64_t* full = reinterpret_cast<uint64_t*>(s_hid + (size_t)NB * h);
  __shared__ float red[NB][kCcScoreThreads / 32][32];
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
  // at most kCcScorePreStages stages before the wait, the rest of the ring
  // right after it (as in the B = 1 scores kernel: a larger early burst
  // delays the wait's return)
  const int first = min(stages, nloc);
  const int pre = min(first, kCcScorePreStages);
  if (threadIdx.x == 0) {
    for (int k = 0; k < pre; ++k) issue(k);
    s_issued = first;
  }
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x == 0)
    for (int k = pre; k < first; ++k) issue(k);
  for (int i = threadIdx.x * 4; i < NB * h; i += kCcScoreThreads * 4)
    *reinterpret_cast<float4*>(s_hid + i) = i < B * h ? ld_dep4(hid + i) : make_float4(0.f, 0.f, 0.f, 0.f);
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
    float acc[NB][32];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int r = 0; r < 32; ++r) acc[b][r] = 0.f;
    for (int c = c0 + lane; c < c1; c += 32) {
      float hv[NB][EPC];
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int e = 0; e < EPC; ++e) hv[b][e] = s_hid[(size_t)b * h + c * EPC + e];
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        float w[EPC];
        WType<T>::unpack(*reinterpret_cast<const uint4*>(sp + (size_t)r * row_bytes + (size_t)c * 16), w);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float t = 0.f;
#pragma unroll
          for (int e = 0; e < EPC; ++e) t = fmaf(w[e], hv[b][e], t);
          acc[b][r] += t;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      cc_transpose_reduce32(acc[b], lane);
      red[b][warp][lane] = acc[b][0];
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (warp == 0) {
      uint32_t u = 0;
      const float bias = b2 ? b2[(size_t)(w0 + k) * 32 + lane] : 0.f;
      for (int b = 0; b < B; ++b) {
        float sc = red[b][0][lane];
#pragma unroll
        for (int w2 = 1; w2 < kCcScoreThreads / 32; ++w2) sc += red[b][w2][lane];
        if (b2) sc += bias;
        const uint32_t m = __ballot_sync(SFFN_FULL_MASK, sc >= thres);  // NaN compares false
        if (lane == 0) nmask[(size_t)b * nw + w0 + k] = m;
        u |= m;
      }
      if (lane == 0) {
        unmask[w0 + k] = u;
        if (k + stages < nloc) {
          fence_proxy_async_smem();
          issue(k + stages);
          s_issued = k + stages + 1;
        }
      }
    }
    __syncthreads();
  }
  if (aborted && threadIdx.x == 0) {
    set_device_error(err, SFFN_ERR_TIMEOUT);
    for (int q = k; q < s_issued; ++q) mbar_wait_bounded(&full[q % stages], (uint32_t)((q / stages) & 1));
  }
}

// The union FFN: as k_ffn (B = 1) over the union list, for B <= NB tokens.
// Each consumer thread owns the 16-byte chunks t, t + 256, ... (at most
// kCcCpt of them, d <= 8192) of every row, so the tokens' x chunks stay in
// registers; one 32 KB ring stage carries as many neurons' up/gate rows (or
// downT rows) as fit.
template <typename T, int ACT, int NB>
__global__ void __launch_bounds__(kCcThreads, 1)
    k_cc_ffn(const T* __restrict__ up, const T* __restrict__ gate, const T* __restrict__ downT, const float* x, int B,
             const uint32_t* nmask, const uint32_t* unmask, int nw, int d, int stages, int list_cap,
             float* __restrict__ partials, uint32_t* __restrict__ err) {
  constexpr int EPC = WType<T>::kPerChunk;
  constexpr bool GATED = act_gated(ACT);
  constexpr int NMAT = GATED ? 2 : 1;
  const uint32_t row_bytes = (uint32_t)(d / EPC) * 16u;
  const int NPS = max(1, (int)(kCcStageBytes / (row_bytes * NMAT)));  // neurons per phase-A stage
  const int RPB = NPS * NMAT;                                        // downT rows per phase-B stage
  const int nch = (int)(row_bytes / 16);

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)stages * kCcStageBytes);
  uint64_t* empty = full + stages;
  uint32_t* s_words = reinterpret_cast<uint32_t*>(empty + stages);    // union words [nw]
  int* s_off = reinterpret_cast<int*>(s_words + nw);
  uint32_t* s_tok = reinterpret_cast<uint32_t*>(s_off + nw);          // token words [NB][nw]
  int32_t* s_list = reinterpret_cast<int32_t*>(s_tok + (size_t)NB * nw);
  float* s_h = reinterpret_cast<float*>(s_list + list_cap);           // [list_cap][NB]
  float* s_part = s_h + (size_t)list_cap * NB;                        // [list_cap][warps][2][NB]
  __shared__ int s_tmp[kCcThreads / 32];
  __shared__ int s_abort;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCcWarps);
    }
    fence_mbar_init();
    s_abort = 0;
  }
  pdl_wait();  // the masks come from the previous kernels
  const int total = scan_mask_words<kCcThreads>(unmask, nw, s_words, s_off, s_tmp);
  for (int i = threadIdx.x; i < NB * nw; i += kCcThreads) s_tok[i] = i < B * nw ? ld_dep(nmask + i) : 0u;
  const int nb = gridDim.x, blk = blockIdx.x;
  const int lo = (int)((long long)total * blk / nb);
  const int hi = (int)((long long)total * (blk + 1) / nb);
  const int n_local = min(hi - lo, list_cap);
  extract_slice<kCcThreads>(s_words, s_off, nw, lo, lo + n_local, s_list);
  __syncthreads();

  const int nA = (n_local + NPS - 1) / NPS;
  const int nB = (n_local + RPB - 1) / RPB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == kCcWarps) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int u = 0; u < nA + nB; ++u) {
        const int s = u % stages;
        const bool ok = u < stages || mbar_wait_bounded(&empty[s], (uint32_t)((u / stages - 1) & 1));
        if (!ok || *(volatile int*)&s_abort) {
          if (!ok) set_device_error(err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
          for (int q = max(0, u - stages); q < u; ++q) mbar_wait_bounded(&full[q % stages], (uint32_t)((q / stages) & 1));
          break;
        }
        unsigned char* dst = ring + (size_t)s * kCcStageBytes;
        if (u < nA) {
          const int k0 = u * NPS, nk = min(NPS, n_local - k0);
          mbar_arrive_expect_tx(&full[s], (uint32_t)nk * NMAT * row_bytes);
          for (int k = 0; k < nk; ++k) {
            const size_t slot = (size_t)s_list[k0 + k];
            unsigned char* dk = dst + (size_t)k * NMAT * row_bytes;
            bulk_g2s(dk, reinterpret_cast<const unsigned char*>(up) + slot * row_bytes, row_bytes, &full[s], pol);
            if (GATED)
              bulk_g2s(dk + row_bytes, reinterpret_cast<const unsigned char*>(gate) + slot * row_bytes, row_bytes,
                       &full[s], pol);
          }
        } else {
          const int r0 = (u - nA) * RPB, nr = min(RPB, n_local - r0);
          mbar_arrive_expect_tx(&full[s], (uint32_t)nr * row_bytes);
          for (int i = 0; i < nr; ++i)
            bulk_g2s(dst + (size_t)i * row_bytes,
                     reinterpret_cast<const unsigned char*>(downT) + (size_t)s_list[r0 + i] * row_bytes, row_bytes,
                     &full[s], pol);
        }
      }
    }
  } else {
    {
      float xr[NB][kCcCpt][EPC];
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int j = 0; j < kCcCpt; ++j) {
          const int c = threadIdx.x + j * kCcConsumers;
#pragma unroll
          for (int e = 0; e < EPC; e += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < nch && b < B) v = ld_dep4(x + (size_t)b * d + (size_t)c * EPC + e);
            xr[b][j][e] = v.x; xr[b][j][e + 1] = v.y; xr[b][j][e + 2] = v.z; xr[b][j][e + 3] = v.w;
          }
        }
      for (int u = 0; u < nA; ++u) {
        const int s = u % stages;
        const bool ok = __all_sync(SFFN_FULL_MASK, mbar_wait_bounded(&full[s], (uint32_t)((u / stages) & 1)));
        if (!ok || __any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
          if (!ok && lane == 0) {
            set_device_error(err, SFFN_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          break;
        }
        const int k0 = u * NPS;
        for (int k = 0; k < NPS; ++k) {
          if (k0 + k >= n_local) break;
          const unsigned char* sp = ring + (size_t)s * kCcStageBytes + (size_t)k * NMAT * row_bytes;
          float pu[NB], pg[NB];
#pragma unroll
          for (int b = 0; b < NB; ++b) pu[b] = pg[b] = 0.f;
#pragma unroll
          for (int j = 0; j < kCcCpt; ++j) {
            const int c = threadIdx.x + j * kCcConsumers;
            if (c < nch) {
              float wu[EPC], wg[EPC];
              WType<T>::unpack(*reinterpret_cast<const uint4*>(sp + (size_t)c * 16), wu);
              if (GATED) WType<T>::unpack(*reinterpret_cast<const uint4*>(sp + row_bytes + (size_t)c * 16), wg);
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                float su = 0.f, sg = 0.f;
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                  su = fmaf(wu[e], xr[b][j][e], su);
                  if (GATED) sg = fmaf(wg[e], xr[b][j][e], sg);
                }
                pu[b] += su;
                if (GATED) pg[b] += sg;
              }
            }
          }
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            pu[b] = warp_sum(pu[b]);
            if (GATED) pg[b] = warp_sum(pg[b]);
          }
          if (lane == 0) {
            float* sp2 = s_part + (((size_t)(k0 + k) * kCcWarps + warp) * 2) * NB;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              sp2[b] = pu[b];
              sp2[NB + b] = pg[b];
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    cc_consumer_barrier();
    // activation per (neuron, token): zero unless the neuron is in the token's own mask
    for (int i = threadIdx.x; i < n_local * NB; i += kCcConsumers) {
      const int a = i / NB, b = i % NB;
      float uu = 0.f, gg = 0.f;
#pragma unroll
      for (int w = 0; w < kCcWarps; ++w) {
        const float* sp2 = s_part + (((size_t)a * kCcWarps + w) * 2) * NB;
        uu += sp2[b];
        gg += sp2[NB + b];
      }
      const int slot = s_list[a];
      const bool mine = (s_tok[(size_t)b * nw + (slot >> 5)] >> (slot & 31)) & 1u;
      s_h[i] = mine ? neuron_act<ACT>(uu, gg) : 0.f;
    }
    cc_consumer_barrier();
    float acc[NB][kCcCpt][EPC];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int j = 0; j < kCcCpt; ++j)
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc[b][j][e] = 0.f;
    if (!__any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
      for (int v = 0; v < nB; ++v) {
        const int u = nA + v;
        const int s = u % stages;
        const bool ok = __all_sync(SFFN_FULL_MASK, mbar_wait_bounded(&full[s], (uint32_t)((u / stages) & 1)));
        if (!ok || __any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
          if (!ok && lane == 0) {
            set_device_error(err, SFFN_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          break;
        }
        const unsigned char* sp = ring + (size_t)s * kCcStageBytes;
        const int r0 = v * RPB, nr = min(RPB, n_local - r0);
        for (int i = 0; i < nr; ++i) {
          float hv[NB];
#pragma unroll
          for (int b = 0; b < NB; ++b) hv[b] = s_h[(size_t)(r0 + i) * NB + b];
#pragma unroll
          for (int j = 0; j < kCcCpt; ++j) {
            const int c = threadIdx.x + j * kCcConsumers;
            if (c < nch) {
              float w[EPC];
              WType<T>::unpack(*reinterpret_cast<const uint4*>(sp + (size_t)i * row_bytes + (size_t)c * 16), w);
#pragma unroll
              for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[b][j][e] = fmaf(hv[b], w[e], acc[b][j][e]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float* part = partials + ((size_t)blk * NB + b) * d;
#pragma unroll
      for (int j = 0; j < kCcCpt; ++j) {
        const int c = threadIdx.x + j * kCcConsumers;
        if (c < nch && b < B) {
#pragma unroll
          for (int e = 0; e < EPC; e += 4)
            *reinterpret_cast<float4*>(part + (size_t)c * EPC + e) =
                make_float4(acc[b][j][e], acc[b][j][e + 1], acc[b][j][e + 2], acc[b][j][e + 3]);
        }
      }
    }
  }
  __syncthreads();
}

// y[b] = sum over blocks of the partials of token b (fixed order), x_out[b] = x[b] + y[b].
template <int PER>
__global__ void __launch_bounds__(kCcReduceThreads)
    k_cc_reduce(const float* partials, int nparts, int NB, int d, const float* x, float* __restrict__ y,
                float* __restrict__ x_out) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int CG = kCcReduceCols / 4;
  constexpr int GROUPS = kCcReduceThreads / CG;
  const int b = blockIdx.y;
  const int cg = threadIdx.x % CG, pg = threadIdx.x / CG;
  const int col = blockIdx.x * kCcReduceCols + cg * 4;
  __shared__ float4 red[GROUPS][CG];
  float4 v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int p = pg + i * GROUPS;
    v[i] = (col < d && p < nparts) ? ld_dep4(partials + ((size_t)p * NB + b) * d + col)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 acc = v[0];
#pragma unroll
  for (int i = 1; i < PER; ++i) {
    acc.x += v[i].x; acc.y += v[i].y; acc.z += v[i].z; acc.w += v[i].w;
  }
  red[pg][cg] = acc;
  __syncthreads();
  if (threadIdx.x < CG && col < d) {
    float4 sum = red[0][cg];
#pragma unroll
    for (int g = 1; g < GROUPS; ++g) {
      const float4 w = red[g][cg];
      sum.x += w.x; sum.y += w.y; sum.z += w.z; sum.w += w.w;
    }
    *reinterpret_cast<float4*>(y + (size_t)b * d + col) = sum;
    if (x_out) {
      const float4 xv = ld_dep4(x + (size_t)b * d + col);
      *reinterpret_cast<float4*>(x_out + (size_t)b * d + col) =
          make_float4(xv.x + sum.x, xv.y + sum.y, xv.z + sum.z, xv.w + sum.w);
    }
  }
}

int cc_hid_cpt(int d) {
  const int nch = d / 8;
  const int need = (nch + kCcHidThreads - 1) / kCcHidThreads;
  return need <= 1 ? 1 : need <= 2 ? 2 : 4;
}

int cc_list_cap(const sffn_layer& L) { return (L.desc.f + L.num_sms - 1) / L.num_sms + 1; }

size_t cc_fixed_smem(const sffn_layer& L, int NB) {
  const size_t cap = (size_t)cc_list_cap(L), nw = (size_t)L.nwords;
  return nw * 8 + (size_t)NB * nw * 4 + cap * 4 + cap * NB * 4 + cap * kCcWarps * 2 * NB * 4;
}

int cc_stages(const sffn_layer& L, int NB) {
  const size_t fixed = cc_fixed_smem(L, NB);
  const size_t budget = (size_t)L.smem_optin > fixed + 2048 ? (size_t)L.smem_optin - fixed - 2048 : 0;
  return (int)std::min<size_t>(8, budget / (kCcStageBytes + 16));
}

size_t cc_ffn_smem(const sffn_layer& L, int NB) {
  return (size_t)cc_stages(L, NB) * (kCcStageBytes + 16) + cc_fixed_smem(L, NB);
}

int cc_score_stages(const sffn_layer& L, int NB) {
  const size_t word = (size_t)32 * L.desc.h * 2;
  const size_t hidb = (size_t)NB * L.desc.h * 4;
  const size_t budget = 192 * 1024 > hidb ? 192 * 1024 - hidb : 0;
  return (int)std::min<size_t>(6, std::max<size_t>(2, budget / word));
}

size_t cc_score_smem(const sffn_layer& L, int NB) {
  return (size_t)cc_score_stages(L, NB) * 32 * L.desc.h * 2 + (size_t)NB * L.desc.h * 4 +
         (size_t)cc_score_stages(L, NB) * 8;
}

int cc_nb(int B) { return B <= 2 ? 2 : 4; }

template <typename T, int NB>
cudaError_t launch_cc_t(const sffn_layer& L, const float* x, int B, float thres, const sffn_masks* m, bool predict,
                        bool forward, float* y, float* x_out, char* base, cudaStream_t st) {
  const BatchCcWs w = batch_cc_ws_layout(L, B);
  const int d = L.desc.d, h = L.desc.h, nw = L.nwords;
  float* hid = reinterpret_cast<float*>(base + w.hid);
  uint32_t* unmask = m->unmask ? m->unmask : reinterpret_cast<uint32_t*>(base + w.unmask);
  int32_t* uidx = m->uidx ? m->uidx : reinterpret_cast<int32_t*>(base + w.uidx);
  int32_t* ucount = m->ucount ? m->ucount : reinterpret_cast<int32_t*>(base + w.ucount);
  float* part = reinterpret_cast<float*>(base + w.partials);
  cudaError_t e = cudaSuccess;
  if (predict) {
    const dim3 hg((h + kCcHidRows - 1) / kCcHidRows), hb(kCcHidThreads);
    const T* W1 = static_cast<const T*>(L.W1);
    const float* b1 = L.has_b1 ? L.b1 : nullptr;
    e = traced_batch(L, 0, st, [&] {
      switch (cc_hid_cpt(d)) {
        case 1: return launch_ex(k_cc_hidden<T, 1, NB>, hg, hb, 0, st, true, 1, W1, b1, x, B, hid, h, d);
        case 2: return launch_ex(k_cc_hidden<T, 2, NB>, hg, hb, 0, st, true, 1, W1, b1, x, B, hid, h, d);
        default: return launch_ex(k_cc_hidden<T, 4, NB>, hg, hb, 0, st, true, 1, W1, b1, x, B, hid, h, d);
      }
    });
    if (e != cudaSuccess) return e;
    const float* b2 = L.has_b2 ? L.b2 : nullptr;
    e = traced_batch(L, 1, st, [&] {
      return launch_ex(k_cc_scores<T, NB>, dim3(std::min(nw, L.num_sms)), dim3(kCcScoreThreads), cc_score_smem(L, NB),
                       st, true, 1, static_cast<const T*>(L.W2), b2, static_cast<const float*>(hid), B, thres,
                       m->nmask, unmask, h, nw, cc_score_stages(L, NB), L.err);
    });
    if (e != cudaSuccess) return e;
  }
  // per-token views (when predicting) and the union views; the union words
  // are already formed when the scores kernel ran
  e = launch_batch_views(L, m, B, unmask, uidx, ucount, predict, predict, st);
  if (e != cudaSuccess || !forward) return e;
  e = traced_batch(L, 2, st, [&] {
    const dim3 grid(L.num_sms), block(kCcThreads);
    const size_t smem = cc_ffn_smem(L, NB);
    const int stages = cc_stages(L, NB), cap = cc_list_cap(L);
    const T* up = static_cast<const T*>(L.up);
    const T* gate = static_cast<const T*>(L.gate);
    const T* dn = static_cast<const T*>(L.downT);
#define SFFN_CC_FFN(A)                                                                                          \
  launch_ex(k_cc_ffn<T, A, NB>, grid, block, smem, st, true, 1, up, gate, dn, x, B,                             \
            static_cast<const uint32_t*>(m->nmask), static_cast<const uint32_t*>(unmask), nw, d, stages, cap, part, \
            L.err)
    switch (L.desc.act) {
      case SFFN_ACT_RELU: return SFFN_CC_FFN(SFFN_ACT_RELU);
      case SFFN_ACT_REGLU: return SFFN_CC_FFN(SFFN_ACT_REGLU);
      case SFFN_ACT_RELU2: return SFFN_CC_FFN(SFFN_ACT_RELU2);
      default: return SFFN_CC_FFN(SFFN_ACT_SWIGLU);
    }
#undef SFFN_CC_FFN
  });
  if (e != cudaSuccess) return e;
  return traced_batch(L, 3, st, [&] {
    const dim3 grid((d + kCcReduceCols - 1) / kCcReduceCols, B), block(kCcReduceThreads);
    const int nparts = L.num_sms, per = (nparts + kCcReduceGroups - 1) / kCcReduceGroups;
    if (per <= 4)
      return launch_ex(k_cc_reduce<4>, grid, block, 0, st, true, 1, static_cast<const float*>(part), nparts, NB, d, x, y,
                       x_out);
    if (per <= 8)
      return launch_ex(k_cc_reduce<8>, grid, block, 0, st, true, 1, static_cast<const float*>(part), nparts, NB, d, x, y,
                       x_out);
    return launch_ex(k_cc_reduce<16>, grid, block, 0, st, true, 1, static_cast<const float*>(part), nparts, NB, d, x, y,
                     x_out);
  });
}

template <typename T>
cudaError_t configure_cc_t(int smem) {
  cudaError_t e;
  if ((e = set_dynamic_smem_max(k_cc_scores<T, 2>, smem))) return e;
  if ((e = set_dynamic_smem_max(k_cc_scores<T, 4>, smem))) return e;
#define SFFN_CC_ATTR(A)                                                   \
  if ((e = set_dynamic_smem_max(k_cc_ffn<T, A, 2>, smem))) return e;      \
  if ((e = set_dynamic_smem_max(k_cc_ffn<T, A, 4>, smem))) return e;
  SFFN_CC_ATTR(SFFN_ACT_RELU)
  SFFN_CC_ATTR(SFFN_ACT_REGLU)
  SFFN_CC_ATTR(SFFN_ACT_SWIGLU)
  SFFN_CC_ATTR(SFFN_ACT_RELU2)
#undef SFFN_CC_ATTR
  return cudaSuccess;
}

}  // namespace

BatchCcWs batch_cc_ws_layout(const sffn_layer& L, int B) {
  auto a256 = [](size_t v) { return (v + 255) & ~size_t(255); };
  const int NB = cc_nb(B);
  BatchCcWs w;
  size_t off = 0;
  w.hid = off;
  off = a256(off + (size_t)NB * L.desc.h * 4);
  w.unmask = off;
  off = a256(off + (size_t)L.nwords * 4);
  w.uidx = off;
  off = a256(off + (size_t)L.desc.f * 4);
  w.ucount = off;
  off = a256(off + 4);
  w.partials = off;
  off = a256(off + (size_t)L.num_sms * NB * L.desc.d * 4);
  w.total = off;
  return w;
}

bool batch_cc_supported(const sffn_layer& L, int B, std::string* why) {
  if (B < 2 || B > kCcMaxBatch) {
    *why = "the CUDA-core batch arm takes 2 to 4 tokens";
    return false;
  }
  if (L.desc.wdtype == SFFN_F32 || L.desc.ffn_format != SFFN_FFN_ROWS) {
    *why = "the CUDA-core batch arm reads 16-bit weights stored as rows";
    return false;
  }
  if (L.desc.d > 256 * kCcCpt * 8) {
    *why = "the CUDA-core batch arm keeps x in registers: d <= 8192";
    return false;
  }
  if ((size_t)L.desc.d * 2 * (act_gated(L.desc.act) ? 2 : 1) > kCcStageBytes) {
    *why = "one neuron's up/gate rows must fit a 32 KB ring stage";
    return false;
  }
  if (cc_stages(L, 4) < 2 || cc_score_smem(L, 4) + 2048 > (size_t)L.smem_optin) {
    *why = "the CUDA-core batch arm's rings do not fit in shared memory for this shape";
    return false;
  }
  return true;
}

cudaError_t configure_batch_cc_kernels(const sffn_layer& L) {
  if (L.desc.wdtype == SFFN_F32) return cudaSuccess;
  return L.desc.wdtype == SFFN_F16 ? configure_cc_t<__half>(L.smem_optin) : configure_cc_t<__nv_bfloat16>(L.smem_optin);
}

cudaError_t launch_batch_cc(const sffn_layer& L, const float* x, int B, float thres, const sffn_masks* m, bool predict,
                            bool forward, float* y, float* x_out, void* ws, cudaStream_t st) {
  char* base = static_cast<char*>(ws);
  const bool bf = L.desc.wdtype == SFFN_BF16;
  if (cc_nb(B) == 2)
    return bf ? launch_cc_t<__nv_bfloat16, 2>(L, x, B, thres, m, predict, forward, y, x_out, base, st)
              : launch_cc_t<__half, 2>(L, x, B, thres, m, predict, forward, y, x_out, base, st);
  return bf ? launch_cc_t<__nv_bfloat16, 4>(L, x, B, thres, m, predict, forward, y, x_out, base, st)
            : launch_cc_t<__half, 4>(L, x, B, thres, m, predict, forward, y, x_out, base, st);
}

}  // namespace sffn
