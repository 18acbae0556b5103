// Neuron-aware sparse FFN (PowerInfer §5.3-§5.4): only the rows of up/gate
// and the transposed-down rows of predicted-active neurons are read.
//
// k_gather_up: each thread block owns a disjoint, contiguous slice of the
//   ascending active list (no cross-block synchronisation). Whole up/gate rows
//   are streamed into a shared-memory ring by one-dimensional bulk copies
//   (TMA), each thread owns fixed 16-byte chunks of the row so its slice of x
//   stays in registers, and the activation is fused into the block reduction.
// k_down: y = sum_i h_i * downT_i. Column slices of d times eight splits of
//   the active list; each block streams its rows' slice chunks through a ring,
//   the eight partial sums of a slice are added through distributed shared
//   memory inside one thread-block cluster, in rank order. No global atomics;
//   the summation order is fixed, so results are bit-identical run to run.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "scan.cuh"

namespace cg = cooperative_groups;

namespace sffn {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kUpThreads = (kConsumerWarps + 1) * 32;    // 8 consumer warps + 1 producer warp
constexpr int kDownThreads = (kConsumerWarps + 1) * 32;
constexpr int kConsumers = kConsumerWarps * 32;

// Gather of the active up/gate rows. Warp 8 is the producer: one lane issues
// the bulk copies of neuron k's rows into ring stage k % S once the consumer
// warps have released that stage (empty barrier, one arrival per warp). The
// eight consumer warps wait for each stage (full barrier, transaction bytes),
// form their partial dot products with the x chunks they own, store one
// partial per warp in shared memory and release the stage; no block-wide
// barrier inside the loop. After the loop the partials of every neuron are
// summed in a fixed order and the activation is applied.
template <typename T, int ACT, int CPT>
__global__ void __launch_bounds__(kUpThreads, 1)
    k_gather_up(const T* __restrict__ up, const T* __restrict__ gate, const float* x,
                const uint32_t* nmask, int nw, int n_groups, int G, int gwords, int d, int stages,
                int list_cap, int32_t* __restrict__ idx_out, int32_t* __restrict__ count_out,
                uint32_t* __restrict__ gmask_out, float* __restrict__ hval, int32_t* __restrict__ alist,
                int32_t* __restrict__ ws_count, uint32_t* __restrict__ err) {
  constexpr int NT = kUpThreads;
  constexpr int EPC = WType<T>::kPerChunk;
  constexpr bool GATED = ACT != SFFN_ACT_RELU;
  const uint32_t row_bytes = (uint32_t)d * sizeof(T);
  const uint32_t stage_bytes = row_bytes * (GATED ? 2u : 1u);
  const int nch = (int)(row_bytes / 16);

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)stages * stage_bytes);
  uint64_t* empty = full + stages;
  uint32_t* s_words = reinterpret_cast<uint32_t*>(empty + stages);
  int* s_off = reinterpret_cast<int*>(s_words + nw);
  int32_t* s_list = reinterpret_cast<int32_t*>(s_off + nw);
  float* s_part = reinterpret_cast<float*>(s_list + list_cap);  // [list_cap][warps][2]
  __shared__ int s_tmp[NT / 32];
  __shared__ int s_abort;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
    s_abort = 0;
  }
  pdl_wait();  // the mask comes from the previous kernel

  const int total = scan_mask_words<NT>(nmask, nw, s_words, s_off, s_tmp);
  const int nb = gridDim.x, b = blockIdx.x;
  const int lo = (int)((long long)total * b / nb);
  const int hi = (int)((long long)total * (b + 1) / nb);
  const int n_local = min(hi - lo, list_cap);
  extract_slice<NT>(s_words, s_off, nw, lo, lo + n_local, s_list);
  if (b == 0) {
    if (threadIdx.x == 0) {
      *ws_count = total;
      if (count_out) *count_out = total;
    }
    if (gmask_out) write_group_mask<NT>(s_words, n_groups, G, gwords, gmask_out);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == kConsumerWarps) {
    // ---------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int k = 0; k < n_local; ++k) {
        const int s = k % stages;
        const bool ok = k < stages || mbar_wait_bounded(&empty[s], (uint32_t)((k / stages - 1) & 1));
        if (!ok || *(volatile int*)&s_abort) {
          if (!ok) set_device_error(err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
          // drain: let the copies that may still be in flight land
          for (int q = max(0, k - stages); q < k; ++q) mbar_wait_bounded(&full[q % stages], (uint32_t)((q / stages) & 1));
          break;
        }
        const size_t slot = (size_t)s_list[k];
        unsigned char* dst = ring + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        bulk_g2s(dst, up + slot * d, row_bytes, &full[s], pol);
        if (GATED) bulk_g2s(dst + row_bytes, gate + slot * d, row_bytes, &full[s], pol);
      }
    }
  } else {
    // ---------------- consumers: this thread's chunks of x, fixed for every row
    float xr[CPT][EPC];
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = threadIdx.x + j * kConsumers;
#pragma unroll
      for (int e = 0; e < EPC; e += 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < nch) v = ld_dep4(x + (size_t)c * EPC + e);
        xr[j][e] = v.x; xr[j][e + 1] = v.y; xr[j][e + 2] = v.z; xr[j][e + 3] = v.w;
      }
    }
    for (int k = 0; k < n_local; ++k) {
      const int s = k % stages;
      // warp-uniform outcome: the shuffles below need every lane
      const bool ok = __all_sync(SFFN_FULL_MASK, mbar_wait_bounded(&full[s], (uint32_t)((k / stages) & 1)));
      if (!ok) {
        if (lane == 0) {
          set_device_error(err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
        break;
      }
      if (__any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) break;
      const unsigned char* sp = ring + (size_t)s * stage_bytes;
      float pu = 0.f, pg = 0.f;
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int c = threadIdx.x + j * kConsumers;
        if (c < nch) {
          pu += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + (size_t)c * 16), xr[j]);
          if (GATED) pg += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + row_bytes + (size_t)c * 16), xr[j]);
        }
      }
      pu = warp_sum(pu);
      if (GATED) pg = warp_sum(pg);
      if (lane == 0) {
        s_part[((size_t)k * kConsumerWarps + warp) * 2] = pu;
        s_part[((size_t)k * kConsumerWarps + warp) * 2 + 1] = pg;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();
  if (s_abort) return;
  for (int k = threadIdx.x; k < n_local; k += NT) {
    float u = 0.f, g = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      u += s_part[((size_t)k * kConsumerWarps + w) * 2];
      g += s_part[((size_t)k * kConsumerWarps + w) * 2 + 1];
    }
    hval[lo + k] = neuron_act<ACT>(u, g);
    const int sl = s_list[k];
    alist[lo + k] = sl;
    if (idx_out) idx_out[lo + k] = sl;
  }
}

// Down projection, y = sum_i h_i * downT_i. Thread-block clusters of eight
// split the active list; the grid's second dimension splits d into column
// slices. The producer warp streams each row's slice chunk into the ring
// (one lane per row); the consumer warps accumulate h_i * chunk in registers
// (each thread owns one 16-byte column chunk and a set of rows) and release
// stages through the empty barriers. Afterwards the row lanes are summed in
// shared memory and the eight blocks' partials are added through distributed
// shared memory in rank order.
template <typename T>
__global__ void __launch_bounds__(kDownThreads, 1)
    k_down(const T* __restrict__ downT, const float* hval, const int32_t* alist,
           const int32_t* ws_count, const float* x, float* __restrict__ y,
           float* __restrict__ x_out, int d, int W, int RS, int stages, int list_cap, uint32_t* __restrict__ err) {
  constexpr int EPC = WType<T>::kPerChunk;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int slice = blockIdx.y;
  const uint32_t chunk_bytes = (uint32_t)W * sizeof(T);
  const int CPR = (int)(chunk_bytes / 16);
  const int RL = kConsumers / CPR;
  const int tc = threadIdx.x % CPR, tr = threadIdx.x / CPR;
  const uint32_t stage_bytes = (uint32_t)RS * chunk_bytes;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + down_region_bytes(W, sizeof(T), RS, stages, kConsumers));
  uint64_t* empty = full + stages;
  float* s_h = reinterpret_cast<float*>(empty + stages);     // [list_cap] this block's h values
  int32_t* s_slot = reinterpret_cast<int32_t*>(s_h + list_cap);  // [list_cap] and their slots
  __shared__ int s_abort;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  pdl_wait();  // h values and the active list come from the previous kernel

  const int total = ld_dep(ws_count);
  const int lo = (int)((long long)total * rank / CL);
  const int hi = (int)((long long)total * (rank + 1) / CL);
  const int n_local = min(hi - lo, list_cap);
  const int nst = (n_local + RS - 1) / RS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t col0 = (size_t)slice * W;
  for (int i = threadIdx.x; i < n_local; i += kDownThreads) {
    s_h[i] = ld_dep(hval + lo + i);
    s_slot[i] = ld_dep(alist + lo + i);
  }
  __syncthreads();

  float acc[EPC];
#pragma unroll
  for (int e = 0; e < EPC; ++e) acc[e] = 0.f;
  if (warp == kConsumerWarps) {
    // ---------------- producer: stage q = rows [q*RS, q*RS + RS), one lane per row
    const uint64_t pol = l2_policy_evict_first();
    for (int q = 0; q < nst; ++q) {
      const int s = q % stages;
      const bool ok = __all_sync(SFFN_FULL_MASK, q < stages || mbar_wait_bounded(&empty[s], (uint32_t)((q / stages - 1) & 1)));
      if (!ok || __any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
        if (lane == 0) {
          if (!ok) set_device_error(err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
          // drain: let the copies that may still be in flight land
          for (int r = max(0, q - stages); r < q; ++r) mbar_wait_bounded(&full[r % stages], (uint32_t)((r / stages) & 1));
        }
        break;
      }
      const int p0 = q * RS;
      const int nr = min(RS, n_local - p0);
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)nr * chunk_bytes);
      __syncwarp();
      if (lane < nr)
        bulk_g2s(ring + (size_t)s * stage_bytes + (size_t)lane * chunk_bytes, downT + (size_t)s_slot[p0 + lane] * d + col0,
                 chunk_bytes, &full[s], pol);
    }
  } else {
    // ---------------- consumers
    for (int q = 0; q < nst; ++q) {
      const int s = q % stages;
      const bool ok = __all_sync(SFFN_FULL_MASK, mbar_wait_bounded(&full[s], (uint32_t)((q / stages) & 1)));
      if (!ok) {
        if (lane == 0) {
          set_device_error(err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
        break;
      }
      if (__any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) break;
      const int p0 = q * RS;
      const int nr = min(RS, n_local - p0);
      if (tr < RL) {
        const unsigned char* sp = ring + (size_t)s * stage_bytes + (size_t)tc * 16;
        for (int r = tr; r < nr; r += RL) {
          const float hv = s_h[p0 + r];
          float w[EPC];
          WType<T>::unpack(*reinterpret_cast<const uint4*>(sp + (size_t)r * chunk_bytes), w);
#pragma unroll
          for (int e = 0; e < EPC; ++e) acc[e] = fmaf(hv, w[e], acc[e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();

  // per-block partial of this column slice: reduce the row lanes in order
  // (the ring region is free once every stage has been consumed)
  float* red = reinterpret_cast<float*>(ring);          // [RL][W]
  float* part = red + (size_t)RL * W;                   // [W]
  if (warp < kConsumerWarps && tr < RL) {
#pragma unroll
    for (int e = 0; e < EPC; ++e) red[(size_t)tr * W + tc * EPC + e] = acc[e];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < W; j += kDownThreads) {
    float sum = 0.f;
    for (int r = 0; r < RL; ++r) sum += red[(size_t)r * W + j];
    part[j] = sum;
  }
  cluster.sync();
  // rank r finishes columns [j0, j1) of the slice, adding the partials of
  // ranks 0..CL-1 in order
  const int j0 = (int)((long long)W * rank / CL), j1 = (int)((long long)W * (rank + 1) / CL);
  for (int j = j0 + threadIdx.x; j < j1; j += kDownThreads) {
    float sum = 0.f;
    for (int r = 0; r < CL; ++r) sum += cluster.map_shared_rank(part, r)[j];
    y[col0 + j] = sum;
    if (x_out) x_out[col0 + j] = ld_dep(x + col0 + j) + sum;
  }
  cluster.sync();
}

template <typename T, int ACT>
cudaError_t launch_up_t(const sffn_layer& L, int cpt, dim3 grid, size_t smem, cudaStream_t st, const float* x,
                        const uint32_t* nmask, int list_cap, int32_t* idx_out, int32_t* count_out,
                        uint32_t* gmask_out, float* hval, int32_t* alist, int32_t* ws_count) {
  const T* up = static_cast<const T*>(L.up);
  const T* gate = static_cast<const T*>(L.gate);
#define SFFN_UP_ARGS                                                                                      \
  grid, dim3(kUpThreads), smem, st, true, 1, up, gate, x, nmask, L.nwords, L.n_groups, L.desc.group_size, \
      L.gwords, L.desc.d, L.up_stages, list_cap, idx_out, count_out, gmask_out, hval, alist, ws_count, L.err
  switch (cpt) {
    case 1: return launch_ex(k_gather_up<T, ACT, 1>, SFFN_UP_ARGS);
    case 2: return launch_ex(k_gather_up<T, ACT, 2>, SFFN_UP_ARGS);
    case 4: return launch_ex(k_gather_up<T, ACT, 4>, SFFN_UP_ARGS);
    default: return launch_ex(k_gather_up<T, ACT, 8>, SFFN_UP_ARGS);
  }
#undef SFFN_UP_ARGS
}

template <typename T, int ACT>
cudaError_t set_up_attr(size_t smem) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_gather_up<T, ACT, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem))) return e;
  if ((e = cudaFuncSetAttribute(k_gather_up<T, ACT, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem))) return e;
  if ((e = cudaFuncSetAttribute(k_gather_up<T, ACT, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem))) return e;
  return cudaFuncSetAttribute(k_gather_up<T, ACT, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

int up_cpt(const sffn_layer& L) {
  const int nch = L.desc.d * L.wbytes / 16;
  const int need = (nch + kConsumers - 1) / kConsumers;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
}

int up_list_cap(const sffn_layer& L) { return (L.desc.f + L.num_sms - 1) / L.num_sms + 1; }

}  // namespace

size_t gather_up_smem(const sffn_layer& L) {
  const size_t row = (size_t)L.desc.d * L.wbytes;
  const size_t stage = row * (L.desc.act == SFFN_ACT_RELU ? 1 : 2);
  return (size_t)L.up_stages * stage + (size_t)L.up_stages * 16 + (size_t)L.nwords * 8 +
         (size_t)up_list_cap(L) * 4 + (size_t)up_list_cap(L) * kConsumerWarps * 2 * 4;
}

int down_list_cap(const sffn_layer& L) { return (L.desc.f + kClusterSplit - 1) / kClusterSplit + 1; }

size_t down_smem(const sffn_layer& L) {
  return down_region_bytes(L.down_width, L.wbytes, L.down_rows_per_stage, L.down_stages, kConsumers) +
         (size_t)L.down_stages * 16 + (size_t)down_list_cap(L) * 8;
}

cudaError_t configure_kernels(sffn_layer& L) {
  const size_t su = gather_up_smem(L), sd = down_smem(L);
  cudaError_t e = cudaSuccess;
  switch (L.desc.wdtype) {
    case SFFN_F32:
      if ((e = set_up_attr<float, SFFN_ACT_RELU>(su)) || (e = set_up_attr<float, SFFN_ACT_REGLU>(su)) ||
          (e = set_up_attr<float, SFFN_ACT_SWIGLU>(su)))
        return e;
      return cudaFuncSetAttribute(k_down<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sd);
    case SFFN_F16:
      if ((e = set_up_attr<__half, SFFN_ACT_RELU>(su)) || (e = set_up_attr<__half, SFFN_ACT_REGLU>(su)) ||
          (e = set_up_attr<__half, SFFN_ACT_SWIGLU>(su)))
        return e;
      return cudaFuncSetAttribute(k_down<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sd);
    default:
      if ((e = set_up_attr<__nv_bfloat16, SFFN_ACT_RELU>(su)) ||
          (e = set_up_attr<__nv_bfloat16, SFFN_ACT_REGLU>(su)) ||
          (e = set_up_attr<__nv_bfloat16, SFFN_ACT_SWIGLU>(su)))
        return e;
      return cudaFuncSetAttribute(k_down<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sd);
  }
}

cudaError_t launch_gather_up(const sffn_layer& L, const float* x, const uint32_t* nmask, int32_t* idx_out,
                             int32_t* count_out, uint32_t* gmask_out, float* hval, int32_t* alist,
                             int32_t* ws_count, cudaStream_t st) {
  const dim3 grid(L.num_sms);
  const size_t smem = gather_up_smem(L);
  const int cpt = up_cpt(L), cap = up_list_cap(L);
#define SFFN_UP_DISPATCH(T)                                                                                   \
  switch (L.desc.act) {                                                                                      \
    case SFFN_ACT_RELU:                                                                                      \
      return launch_up_t<T, SFFN_ACT_RELU>(L, cpt, grid, smem, st, x, nmask, cap, idx_out, count_out,         \
                                           gmask_out, hval, alist, ws_count);                                \
    case SFFN_ACT_REGLU:                                                                                     \
      return launch_up_t<T, SFFN_ACT_REGLU>(L, cpt, grid, smem, st, x, nmask, cap, idx_out, count_out,        \
                                            gmask_out, hval, alist, ws_count);                               \
    default:                                                                                                 \
      return launch_up_t<T, SFFN_ACT_SWIGLU>(L, cpt, grid, smem, st, x, nmask, cap, idx_out, count_out,       \
                                             gmask_out, hval, alist, ws_count);                              \
  }
  switch (L.desc.wdtype) {
    case SFFN_F32: SFFN_UP_DISPATCH(float)
    case SFFN_F16: SFFN_UP_DISPATCH(__half)
    default: SFFN_UP_DISPATCH(__nv_bfloat16)
  }
#undef SFFN_UP_DISPATCH
}

cudaError_t launch_down(const sffn_layer& L, const float* hval, const int32_t* alist, const int32_t* ws_count,
                        const float* x, float* y, float* x_out, cudaStream_t st) {
  const dim3 grid(kClusterSplit, L.down_slices);
  const size_t smem = down_smem(L);
#define SFFN_DOWN_ARGS                                                                                     \
  grid, dim3(kDownThreads), smem, st, true, kClusterSplit, static_cast<const T*>(L.downT), hval, alist,    \
      ws_count, x, y, x_out, L.desc.d, L.down_width, L.down_rows_per_stage, L.down_stages, down_list_cap(L), L.err
  switch (L.desc.wdtype) {
    case SFFN_F32: {
      using T = float;
      return launch_ex(k_down<T>, SFFN_DOWN_ARGS);
    }
    case SFFN_F16: {
      using T = __half;
      return launch_ex(k_down<T>, SFFN_DOWN_ARGS);
    }
    default: {
      using T = __nv_bfloat16;
      return launch_ex(k_down<T>, SFFN_DOWN_ARGS);
    }
  }
#undef SFFN_DOWN_ARGS
}

}  // namespace sffn
