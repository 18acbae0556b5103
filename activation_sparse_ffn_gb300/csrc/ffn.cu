// Neuron-aware sparse FFN (PowerInfer §5.3-§5.4): only the rows of up/gate
// and the transposed-down rows of predicted-active neurons are read, and each
// thread block owns a disjoint, contiguous slice of the ascending active list
// (no cross-block synchronisation inside the kernel).
//
// k_ffn streams, per block, first the up (and gate) rows of its neurons and
// then their downT rows through one shared-memory ring of whole-row
// one-dimensional bulk copies (TMA). Warp 8 is the producer (one lane issues
// the copies once the eight consumer warps have released a stage through its
// empty barrier); the consumer warps wait on the stage's full barrier
// (transaction bytes). Phase A: each consumer thread owns fixed 16-byte chunks
// of a row, so its slice of x stays in registers; one partial dot product per
// warp and neuron goes to shared memory. After one barrier among the
// consumers the partials of every neuron are summed in a fixed order and the
// activation gives h. Phase B: the same chunk ownership accumulates
// h_i * downT_i into per-thread registers, so the block ends with a partial of
// y over its neurons, written to the workspace.
// Zero-skip (optional): the consumers list the local neurons whose h is not
// zero and publish the list through an mbarrier; the producer streams phase B
// over that list only (a neuron with h = 0 adds nothing to y).
// k_ffn_reduce adds the blocks' partials in a fixed order (no atomics) and
// writes y and the residual x + y. Results are bit-identical run to run.
#include "common.cuh"
#include "internal.h"
#include "scan.cuh"

#include <algorithm>
#include <type_traits>

namespace sffn {

namespace {

constexpr int kConsumerWarps = 8;

// Neurons per ring stage for FFN weights of `bits` bits whose rows take `cpt`
// 16-byte chunks per consumer thread (a row is at most cpt x 4 KB), `nmat`
// rows per neuron in phase A. A stage costs a roughly fixed time on top of its
// bytes, so 16- and 32-bit rows travel as many neurons to a stage as fill a
// target size: 32 KB for rows over 8 KB, 64 KB for shorter rows. Measured on
// GB300: random 8 KB rows stream at 31 GB/s per SM through 16 KB stages and
// at 42 through 32 KB stages (the same bytes in flight); 64 KB stages made
// the 8 KB-row layers 7% (sparse SwiGLU) and 13% (dense) faster, and left the
// sparse 16 KB-row layers unchanged or 0.5% slower. The
// quantized formats take 4 (8-bit) or 8 (4-bit) neurons. Host and device take
// the ring's stage size from this one rule.
__host__ __device__ constexpr int neurons_per_stage(int bits, int cpt, int nmat) {
  return bits == 8 ? 4 : bits == 4 ? 8 : nmat * cpt >= (cpt <= 2 ? 16 : 8) ? 1 : (cpt <= 2 ? 16 : 8) / (nmat * cpt);
}
constexpr int kFfnThreads = (kConsumerWarps + 1) * 32;  // 8 consumer warps + 1 producer warp
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kReduceThreads = 256;
constexpr int kReduceCols = 32;                          // columns per reduction block
constexpr int kReduceGroups = kReduceThreads / (kReduceCols / 4);  // 32 partial groups

__device__ __forceinline__ void consumer_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Block b's share (1/nb, 16-byte granules) of [base, base + bytes), handed to
// L2 as bulk prefetches of at most 64 KB.
__device__ __forceinline__ void prefetch_share(const unsigned char* base, size_t bytes, int b, int nb) {
  if (!base) return;
  const size_t units = bytes / 16;
  const size_t lo = units * (size_t)b / (size_t)nb * 16, hi = units * (size_t)(b + 1) / (size_t)nb * 16;
  for (size_t o = lo; o < hi; o += 65536) prefetch_l2_bulk(base + o, (uint32_t)min(hi - o, (size_t)65536));
}

template <typename T, int ACT, int CPT>
__global__ void __launch_bounds__(kFfnThreads, 1)
    k_ffn(const T* __restrict__ up, const T* __restrict__ gate, const T* __restrict__ downT, const float* x,
          const uint32_t* nmask, int nw, int n_groups, int G, int gwords, int d, int stages, int list_cap,
          int32_t* __restrict__ idx_out, int32_t* __restrict__ count_out, uint32_t* __restrict__ gmask_out,
          float* __restrict__ partials, uint32_t* __restrict__ err, const unsigned char* pf, size_t pf_bytes,
          const float* __restrict__ up_s, const float* __restrict__ gate_s, const float* __restrict__ down_s,
          const uint32_t* resident, bool zero_skip, int32_t* __restrict__ kept) {
  constexpr int NT = kFfnThreads;
  constexpr int EPC = WType<T>::kPerChunk;
  constexpr bool GATED = act_gated(ACT);
  // 8-bit and 4-bit rows: codes times one scale per neuron (up_s, gate_s, down_s)
  constexpr bool QS = std::is_same<T, int8_t>::value || std::is_same<T, q4x2_t>::value;
  constexpr int NMAT = GATED ? 2 : 1;  // rows per neuron in phase A
  constexpr int NPS = neurons_per_stage(128 / EPC, CPT, NMAT);  // a 16-byte chunk holds EPC weights
  const uint32_t row_bytes = (uint32_t)(d / EPC) * 16u;
  const uint32_t stage_bytes = row_bytes * NMAT * NPS;
  const int nch = (int)(row_bytes / 16);

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)stages * stage_bytes);
  uint64_t* empty = full + stages;
  uint32_t* s_words = reinterpret_cast<uint32_t*>(empty + stages);
  int* s_off = reinterpret_cast<int*>(s_words + nw);
  int32_t* s_list = reinterpret_cast<int32_t*>(s_off + nw);
  float* s_h = reinterpret_cast<float*>(s_list + list_cap);
  float* s_part = s_h + list_cap;  // [list_cap][warps][2]
  __shared__ int s_tmp[NT / 32];
  __shared__ int s_abort;
  __shared__ uint32_t s_res[32];  // L2-resident groups (at most 1024)
  __shared__ uint64_t s_hready;    // zero-skip: the kept list is published
  __shared__ int s_nkeep;          // zero-skip: neurons in the kept list
  __shared__ int s_wcnt[kConsumerWarps];

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&s_hready, 1);
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
  // the optional hot-group set (may be written by the previous kernel)
  if (threadIdx.x < 32) s_res[threadIdx.x] = (resident && (int)threadIdx.x < gwords) ? ld_dep(resident + threadIdx.x) : 0u;
  if (b == 0) {
    if (threadIdx.x == 0 && count_out) *count_out = total;
    if (gmask_out) write_group_mask<NT>(s_words, n_groups, G, gwords, gmask_out);
  }
  __syncthreads();

  const int nA = (n_local + NPS - 1) / NPS;                  // phase A stages: NPS neurons' up [+ gate]
  const int nB = (n_local + NMAT * NPS - 1) / (NMAT * NPS);  // phase B stages: NMAT * NPS downT rows
  // zero-skip: phase B reads the rows of the kept list, written over s_part
  // once the activations are known (s_part is not read after that)
  const int32_t* s_keep = reinterpret_cast<const int32_t*>(s_part);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == kConsumerWarps) {
    // ---------------- producer
    if (lane == 0) {
      // rows of hot groups stay in L2 for the next tokens, the rest streams through
      const uint64_t pol_stream = l2_policy_evict_first(), pol_keep = l2_policy_keep();
      auto pol_of = [&](int slot) {
        const int g = slot / G;
        return (s_res[g >> 5] >> (g & 31)) & 1u ? pol_keep : pol_stream;
      };
      int nBp = nB;  // zero-skip: known once the consumers publish the kept list
      for (int u = 0; u < nA + nBp; ++u) {
        const int s = u % stages;
        bool ok = true;
        if (zero_skip && u == nA) {
          ok = mbar_wait_bounded(&s_hready, 0u);
          if (ok) {
            nBp = (*(volatile int*)&s_nkeep + NMAT * NPS - 1) / (NMAT * NPS);
            if (nBp == 0) break;
          }
        }
        ok = ok && (u < stages || mbar_wait_bounded(&empty[s], (uint32_t)((u / stages - 1) & 1)));
        if (!ok || *(volatile int*)&s_abort) {
          if (!ok) set_device_error(err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
          // drain: let the copies that may still be in flight land
          for (int q = max(0, u - stages); q < u; ++q) mbar_wait_bounded(&full[q % stages], (uint32_t)((q / stages) & 1));
          break;
        }
        unsigned char* dst = ring + (size_t)s * stage_bytes;
        if (u < nA) {
          const int k0 = u * NPS, nk = min(NPS, n_local - k0);
          mbar_arrive_expect_tx(&full[s], (uint32_t)nk * NMAT * row_bytes);
          for (int k = 0; k < nk; ++k) {
            const size_t slot = (size_t)s_list[k0 + k];
            const uint64_t pol = pol_of((int)slot);
            unsigned char* dk = dst + (size_t)k * NMAT * row_bytes;
            bulk_g2s(dk, reinterpret_cast<const unsigned char*>(up) + slot * row_bytes, row_bytes, &full[s], pol);
            if (GATED)
              bulk_g2s(dk + row_bytes, reinterpret_cast<const unsigned char*>(gate) + slot * row_bytes, row_bytes,
                       &full[s], pol);
          }
        } else {
          const int r0 = (u - nA) * NMAT * NPS;
          const int nr = min(NMAT * NPS, (zero_skip ? *(volatile int*)&s_nkeep : n_local) - r0);
          mbar_arrive_expect_tx(&full[s], (uint32_t)nr * row_bytes);
          for (int i = 0; i < nr; ++i) {
            const int slot = s_list[zero_skip ? s_keep[r0 + i] : r0 + i];
            bulk_g2s(dst + (size_t)i * row_bytes, reinterpret_cast<const unsigned char*>(downT) + (size_t)slot * row_bytes,
                     row_bytes, &full[s], pol_of(slot));
          }
        }
      }
      // L2 hint: once this block's rows are all requested, its share of the
      // next layer's predictor hidden-layer weights (pf is null without a hint)
      if (!*(volatile int*)&s_abort) prefetch_share(pf, pf_bytes, b, nb);
    }
  } else {
    // ---------------- consumers, phase A: partial dot products of up/gate rows
    // (coded rows hold x as pairs for packed fp32 arithmetic: their dequantization
    // makes them issue-bound, not bandwidth-bound)
    {
      float xr[CPT][QS ? 1 : EPC];
      float2 xp[CPT][QS ? EPC / 2 : 1];
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int c = threadIdx.x + j * kConsumers;
#pragma unroll
        for (int e = 0; e < EPC; e += 4) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (c < nch) v = ld_dep4(x + (size_t)c * EPC + e);
          if constexpr (QS) {
            xp[j][e / 2] = make_float2(v.x, v.y);
            xp[j][e / 2 + 1] = make_float2(v.z, v.w);
          } else {
            xr[j][e] = v.x; xr[j][e + 1] = v.y; xr[j][e + 2] = v.z; xr[j][e + 3] = v.w;
          }
        }
      }
      for (int u = 0; u < nA; ++u) {
        const int s = u % stages;
        // warp-uniform outcome: the shuffles below need every lane
        const bool ok = __all_sync(SFFN_FULL_MASK, mbar_wait_bounded(&full[s], (uint32_t)((u / stages) & 1)));
        if (!ok || __any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
          if (!ok && lane == 0) {
            set_device_error(err, SFFN_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          break;
        }
        const int k0 = u * NPS;
#pragma unroll
        for (int k = 0; k < NPS; ++k) {
          if (k0 + k >= n_local) break;
          const unsigned char* sp = ring + (size_t)s * stage_bytes + (size_t)k * NMAT * row_bytes;
          float pu = 0.f, pg = 0.f;
#pragma unroll
          for (int j = 0; j < CPT; ++j) {
            const int c = threadIdx.x + j * kConsumers;
            if (c < nch) {
              const uint4 wu = *reinterpret_cast<const uint4*>(sp + (size_t)c * 16);
              if constexpr (QS) {
                pu += dot_chunk_pairs<T>(wu, xp[j]);
                if (GATED) pg += dot_chunk_pairs<T>(*reinterpret_cast<const uint4*>(sp + row_bytes + (size_t)c * 16), xp[j]);
              } else {
                pu += dot_chunk<T>(wu, xr[j]);
                if (GATED) pg += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + row_bytes + (size_t)c * 16), xr[j]);
              }
            }
          }
          pu = warp_sum(pu);
          if (GATED) pg = warp_sum(pg);
          if (lane == 0) {
            s_part[((size_t)(k0 + k) * kConsumerWarps + warp) * 2] = pu;
            s_part[((size_t)(k0 + k) * kConsumerWarps + warp) * 2 + 1] = pg;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    consumer_barrier();
    // activation of every local neuron, partials added in warp order
    for (int a = threadIdx.x; a < n_local; a += kConsumers) {
      float uu = 0.f, gg = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        uu += s_part[((size_t)a * kConsumerWarps + w) * 2];
        gg += s_part[((size_t)a * kConsumerWarps + w) * 2 + 1];
      }
      if (QS) {
        const int slot = s_list[a];
        uu *= up_s[slot];
        if (GATED) gg *= gate_s[slot];
        // phase B multiplies the downT codes by h x the neuron's down scale
        s_h[a] = neuron_act<ACT>(uu, gg) * down_s[slot];
      } else {
        s_h[a] = neuron_act<ACT>(uu, gg);
      }
      if (idx_out) idx_out[lo + a] = s_list[a];
    }
    consumer_barrier();
    int nkeep = n_local;  // neurons phase B reads
    if (zero_skip) {
      // the kept list: local neurons with h != 0 (NaN kept), ascending
      int32_t* keep = reinterpret_cast<int32_t*>(s_part);
      nkeep = 0;
      for (int base = 0; base < n_local; base += kConsumers) {
        const int a = base + threadIdx.x;
        const bool k = a < n_local && s_h[a] != 0.f;
        const uint32_t bal = __ballot_sync(SFFN_FULL_MASK, k);
        if (lane == 0) s_wcnt[warp] = __popc(bal);
        consumer_barrier();
        int off = nkeep, tot = 0;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          off += w < warp ? s_wcnt[w] : 0;
          tot += s_wcnt[w];
        }
        if (k) keep[off + __popc(bal & ((1u << lane) - 1u))] = a;
        nkeep += tot;
        consumer_barrier();
      }
      if (threadIdx.x == 0) {
        s_nkeep = nkeep;
        if (kept) kept[b] = nkeep;
        mbar_arrive(&s_hready);  // release: the list and its length to the producer
      }
    }
    const int nBc = (nkeep + NMAT * NPS - 1) / (NMAT * NPS);
    // ---------------- phase B: acc += h_i * downT_i over this block's neurons
    float acc[CPT][QS ? 1 : EPC];
    float2 accp[CPT][QS ? EPC / 2 : 1];  // coded rows: pairs
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
#pragma unroll
      for (int e = 0; e < (QS ? 1 : EPC); ++e) acc[j][e] = 0.f;
#pragma unroll
      for (int e = 0; e < (QS ? EPC / 2 : 1); ++e) accp[j][e] = make_float2(0.f, 0.f);
    }
    if (!__any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
      for (int v = 0; v < nBc; ++v) {
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
        const unsigned char* sp = ring + (size_t)s * stage_bytes;
        const int r0 = v * NMAT * NPS;
        const int nr = min(NMAT * NPS, nkeep - r0);
        for (int i = 0; i < nr; ++i) {
          const float hv = s_h[zero_skip ? s_keep[r0 + i] : r0 + i];
#pragma unroll
          for (int j = 0; j < CPT; ++j) {
            const int c = threadIdx.x + j * kConsumers;
            if (c < nch) {
              const uint4 wv = *reinterpret_cast<const uint4*>(sp + (size_t)i * row_bytes + (size_t)c * 16);
              if constexpr (QS) {
                float2 w[EPC / 2];
                WType<T>::unpack2(wv, w);
                const float2 h2 = make_float2(hv, hv);
#pragma unroll
                for (int e = 0; e < EPC / 2; ++e) accp[j][e] = __ffma2_rn(h2, w[e], accp[j][e]);
              } else {
                float w[EPC];
                WType<T>::unpack(wv, w);
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[j][e] = fmaf(hv, w[e], acc[j][e]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    // this block's partial of y
    float* part = partials + (size_t)b * d;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = threadIdx.x + j * kConsumers;
      if (c < nch) {
#pragma unroll
        for (int e = 0; e < EPC; e += 4) {
          if constexpr (QS)
            *reinterpret_cast<float4*>(part + (size_t)c * EPC + e) =
                make_float4(accp[j][e / 2].x, accp[j][e / 2].y, accp[j][e / 2 + 1].x, accp[j][e / 2 + 1].y);
          else
            *reinterpret_cast<float4*>(part + (size_t)c * EPC + e) =
                make_float4(acc[j][e], acc[j][e + 1], acc[j][e + 2], acc[j][e + 3]);
        }
      }
    }
  }
  __syncthreads();
}

// y = sum over blocks of the partials; x_out = x + y. Each block covers
// kReduceCols columns with kReduceGroups groups of threads, group g adding
// the partials g, g + kReduceGroups, ... (all loads of a thread issued before
// any add); the group sums are then added in group order. Fixed order, no
// atomics.
template <int PER>
__global__ void __launch_bounds__(kReduceThreads)
    k_ffn_reduce(const float* partials, int nparts, int d, const float* x, float* __restrict__ y,
                 float* __restrict__ x_out, const int32_t* kept, int32_t* __restrict__ rows_read) {
  pdl_launch_dependents();
  pdl_wait();  // the partials come from the previous kernel
  constexpr int CG = kReduceCols / 4;             // float4 column groups per block
  constexpr int GROUPS = kReduceThreads / CG;     // partial groups
  const int cg = threadIdx.x % CG, pg = threadIdx.x / CG;
  const int col = blockIdx.x * kReduceCols + cg * 4;
  __shared__ float4 red[GROUPS][CG];
  // the residual's x, requested together with the partials (one round trip)
  const bool adds = threadIdx.x < CG && col < d;
  const float4 xv = (x_out && adds) ? ld_dep4(x + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int p = pg + i * GROUPS;
    v[i] = (col < d && p < nparts) ? ld_dep4(partials + (size_t)p * d + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 acc = v[0];
#pragma unroll
  for (int i = 1; i < PER; ++i) {
    acc.x += v[i].x; acc.y += v[i].y; acc.z += v[i].z; acc.w += v[i].w;
  }
  red[pg][cg] = acc;
  __syncthreads();
  if (adds) {
    float4 sum = red[0][cg];
#pragma unroll
    for (int g = 1; g < GROUPS; ++g) {
      const float4 w = red[g][cg];
      sum.x += w.x; sum.y += w.y; sum.z += w.z; sum.w += w.w;
    }
    *reinterpret_cast<float4*>(y + col) = sum;
    if (x_out)
      *reinterpret_cast<float4*>(x_out + col) = make_float4(xv.x + sum.x, xv.y + sum.y, xv.z + sum.z, xv.w + sum.w);
  }
  // zero-skip: the downT rows the FFN blocks read (one warp of the last block;
  // an integer sum, so its order does not matter)
  if (rows_read && blockIdx.x == gridDim.x - 1 && threadIdx.x < 32) {
    int n = 0;
    for (int i = threadIdx.x; i < nparts; i += 32) n += ld_dep(kept + i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(SFFN_FULL_MASK, n, o);
    if (threadIdx.x == 0) *rows_read = n;
  }
}

// Largest chunk count per consumer thread a row of type T can need: rows are
// at most 32 KB of 16- or 32-bit weights (8 chunks per thread), so at most
// 16 KB of 8-bit codes (4) and 8 KB of 4-bit codes (2). Only these
// instantiations are built.
template <typename T>
constexpr int max_ffn_cpt() {
  return std::is_same<T, q4x2_t>::value ? 2 : std::is_same<T, int8_t>::value ? 4 : 8;
}

template <typename T, int ACT>
cudaError_t launch_ffn_t(const sffn_layer& L, int cpt, dim3 grid, size_t smem, cudaStream_t st, const float* x,
                         const uint32_t* nmask, int list_cap, int32_t* idx_out, int32_t* count_out,
                         uint32_t* gmask_out, float* partials, int32_t* kept) {
  const T* up = static_cast<const T*>(L.up);
  const T* gate = static_cast<const T*>(L.gate);
  const T* downT = static_cast<const T*>(L.downT);
  // The optional L2 hint: the next layer's W1 only. Its 16.8 MB (70B shape)
  // fit the HBM time that this kernel's tail and the reduction leave idle;
  // adding W2 as well competed with this kernel's own row stream and lost.
  const sffn_layer* nx = L.next;
  const unsigned char* pf = nx ? static_cast<const unsigned char*>(nx->W1) : nullptr;
  const size_t pf_bytes = nx ? (size_t)nx->desc.h * nx->desc.d * nx->wbytes : 0;
#define SFFN_FFN_ARGS                                                                                         \
  grid, dim3(kFfnThreads), smem, st, true, 1, up, gate, downT, x, nmask, L.nwords, L.n_groups,                \
      L.desc.group_size, L.gwords, L.desc.d, L.ffn_stages, list_cap, idx_out, count_out, gmask_out, partials, L.err, pf, pf_bytes, L.up_s, L.gate_s, L.down_s, \
      L.l2_resident, L.zero_skip, L.zero_skip ? kept : nullptr
  switch (cpt) {
    case 1: return launch_ex(k_ffn<T, ACT, 1>, SFFN_FFN_ARGS);
    case 2: return launch_ex(k_ffn<T, ACT, 2>, SFFN_FFN_ARGS);
    case 4:
      if constexpr (max_ffn_cpt<T>() >= 4) return launch_ex(k_ffn<T, ACT, 4>, SFFN_FFN_ARGS);
      return cudaErrorInvalidConfiguration;
    default:
      if constexpr (max_ffn_cpt<T>() >= 8) return launch_ex(k_ffn<T, ACT, 8>, SFFN_FFN_ARGS);
      return cudaErrorInvalidConfiguration;
  }
#undef SFFN_FFN_ARGS
}

template <typename K>
cudaError_t set_big_smem(K* kern, size_t smem) {
  cudaError_t e = set_dynamic_smem_max(kern, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

template <typename T, int ACT>
cudaError_t set_ffn_attr(size_t smem) {
  cudaError_t e;
  if ((e = set_big_smem(k_ffn<T, ACT, 1>, smem))) return e;
  if ((e = set_big_smem(k_ffn<T, ACT, 2>, smem))) return e;
  if constexpr (max_ffn_cpt<T>() >= 4)
    if ((e = set_big_smem(k_ffn<T, ACT, 4>, smem))) return e;
  if constexpr (max_ffn_cpt<T>() >= 8) return set_big_smem(k_ffn<T, ACT, 8>, smem);
  return cudaSuccess;
}

int ffn_cpt(const sffn_layer& L) {
  const int nch = (int)(ffn_row_bytes(L) / 16);
  const int need = (nch + kConsumers - 1) / kConsumers;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
}

int ffn_grid_of(const sffn_layer& L) { return L.ffn_grid > 0 ? L.ffn_grid : L.num_sms; }
int ffn_list_cap(const sffn_layer& L) { return (L.desc.f + ffn_grid_of(L) - 1) / ffn_grid_of(L) + 1; }

size_t ffn_fixed_smem(const sffn_layer& L) {
  const size_t cap = (size_t)ffn_list_cap(L);
  return (size_t)L.nwords * 8 + cap * 4 + cap * 4 + cap * kConsumerWarps * 2 * 4;
}

}  // namespace

cudaError_t set_max_carveout();

int ffn_blocks(const sffn_layer& L) { return ffn_grid_of(L); }

int ffn_stages_for(const sffn_layer& L) {
  const size_t stage = ffn_row_bytes(L) * (act_gated(L.desc.act) ? 2 : 1) *
                       neurons_per_stage(L.fbits, ffn_cpt(L), act_gated(L.desc.act) ? 2 : 1);
  const size_t budget = kFfnSmemBudget > ffn_fixed_smem(L) ? kFfnSmemBudget - ffn_fixed_smem(L) : 0;
  return (int)std::min<size_t>(kFfnMaxStages, budget / (stage + 16));
}

size_t ffn_smem(const sffn_layer& L) {
  const size_t stage = ffn_row_bytes(L) * (act_gated(L.desc.act) ? 2 : 1) *
                       neurons_per_stage(L.fbits, ffn_cpt(L), act_gated(L.desc.act) ? 2 : 1);
  return (size_t)L.ffn_stages * (stage + 16) + ffn_fixed_smem(L);
}

// Kernel attributes are shared by every layer in the process, so the dynamic
// shared-memory limit is raised to the device maximum once rather than to
// this layer's need (a smaller layer created later must not lower it).
cudaError_t configure_kernels(sffn_layer& L) {
  if (ffn_smem(L) + 1024 > (size_t)L.smem_optin) return cudaErrorInvalidConfiguration;
  const size_t sm = (size_t)L.smem_optin;
  cudaError_t e = set_max_carveout();
  if (e != cudaSuccess) return e;
#define SFFN_FFN_ATTRS(T)                                                                                   \
  if ((e = set_ffn_attr<T, SFFN_ACT_RELU>(sm)) || (e = set_ffn_attr<T, SFFN_ACT_REGLU>(sm)) ||              \
      (e = set_ffn_attr<T, SFFN_ACT_SWIGLU>(sm)))                                                            \
    return e;                                                                                                \
  return set_ffn_attr<T, SFFN_ACT_RELU2>(sm);
  if (L.desc.ffn_format == SFFN_FFN_Q4) {
    SFFN_FFN_ATTRS(q4x2_t)
  }
  if (L.desc.ffn_format == SFFN_FFN_Q8) {
    SFFN_FFN_ATTRS(int8_t)
  }
  switch (L.desc.wdtype) {
    case SFFN_F32: SFFN_FFN_ATTRS(float)
    case SFFN_F16: SFFN_FFN_ATTRS(__half)
    default: SFFN_FFN_ATTRS(__nv_bfloat16)
  }
#undef SFFN_FFN_ATTRS
}


cudaError_t launch_ffn(const sffn_layer& L, const float* x, const uint32_t* nmask, int32_t* idx_out,
                       int32_t* count_out, uint32_t* gmask_out, float* partials, int32_t* kept, cudaStream_t st) {
  const dim3 grid(ffn_blocks(L));
  const size_t smem = ffn_smem(L);
  const int cpt = ffn_cpt(L), cap = ffn_list_cap(L);
#define SFFN_FFN_DISPATCH(T)                                                                                  \
  switch (L.desc.act) {                                                                                      \
    case SFFN_ACT_RELU:                                                                                      \
      return launch_ffn_t<T, SFFN_ACT_RELU>(L, cpt, grid, smem, st, x, nmask, cap, idx_out, count_out,        \
                                            gmask_out, partials, kept);               \
    case SFFN_ACT_REGLU:                                                                                     \
      return launch_ffn_t<T, SFFN_ACT_REGLU>(L, cpt, grid, smem, st, x, nmask, cap, idx_out, count_out,       \
                                             gmask_out, partials, kept);              \
    case SFFN_ACT_RELU2:                                                                                     \
      return launch_ffn_t<T, SFFN_ACT_RELU2>(L, cpt, grid, smem, st, x, nmask, cap, idx_out, count_out,       \
                                             gmask_out, partials, kept);              \
    default:                                                                                                 \
      return launch_ffn_t<T, SFFN_ACT_SWIGLU>(L, cpt, grid, smem, st, x, nmask, cap, idx_out, count_out,      \
                                              gmask_out, partials, kept);             \
  }
  if (L.desc.ffn_format == SFFN_FFN_Q4) {
    SFFN_FFN_DISPATCH(q4x2_t)
  }
  if (L.desc.ffn_format == SFFN_FFN_Q8) {
    SFFN_FFN_DISPATCH(int8_t)
  }
  switch (L.desc.wdtype) {
    case SFFN_F32: SFFN_FFN_DISPATCH(float)
    case SFFN_F16: SFFN_FFN_DISPATCH(__half)
    default: SFFN_FFN_DISPATCH(__nv_bfloat16)
  }
#undef SFFN_FFN_DISPATCH
}

cudaError_t launch_ffn_reduce(const sffn_layer& L, const float* partials, const int32_t* kept, const float* x,
                              float* y, float* x_out, cudaStream_t st) {
  const dim3 grid((L.desc.d + kReduceCols - 1) / kReduceCols), block(kReduceThreads);
  const int nparts = ffn_blocks(L);
  const int per = (nparts + kReduceGroups - 1) / kReduceGroups;
  int32_t* rows_read = L.zero_skip ? L.rows_read : nullptr;
  if (per <= 4)
    return launch_ex(k_ffn_reduce<4>, grid, block, 0, st, true, 1, partials, nparts, L.desc.d, x, y, x_out, kept,
                     rows_read);
  if (per <= 8)
    return launch_ex(k_ffn_reduce<8>, grid, block, 0, st, true, 1, partials, nparts, L.desc.d, x, y, x_out, kept,
                     rows_read);
  if (per <= 16)
    return launch_ex(k_ffn_reduce<16>, grid, block, 0, st, true, 1, partials, nparts, L.desc.d, x, y, x_out, kept,
                     rows_read);
  return cudaErrorNotSupported;  // more than 512 blocks: not reached on current GPUs
}

cudaError_t set_max_carveout() {
  // Every hot kernel asks for the largest shared-memory carveout, so that
  // consecutive kernels of a decode step need no L1/shared reconfiguration.
  cudaError_t e;
  const int c = cudaSharedmemCarveoutMaxShared;
  if ((e = cudaFuncSetAttribute(k_ffn_reduce<4>, cudaFuncAttributePreferredSharedMemoryCarveout, c))) return e;
  if ((e = cudaFuncSetAttribute(k_ffn_reduce<8>, cudaFuncAttributePreferredSharedMemoryCarveout, c))) return e;
  return cudaFuncSetAttribute(k_ffn_reduce<16>, cudaFuncAttributePreferredSharedMemoryCarveout, c);
}

}  // namespace sffn
