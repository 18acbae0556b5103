// One decode token through a whole stack of layers in one persistent kernel
// (B = 1): for every layer, the predictor (PowerInfer §5.1: hidden layer,
// scores, threshold), the neuron-aware sparse FFN on the predicted set
// (§5.3-§5.4) and the residual x_{l+1} = x_l + y_l.
//
// One thread block per SM; 8 consumer warps and 1 producer warp. The
// producer streams, through one shared-memory ring of 32 KB stages filled by
// one-dimensional bulk copies (TMA), every byte the block's consumers will
// read, in the order they read it:
//   per layer  H  its share of the predictor's W1 rows,
//              S  its share of W2 (whole 32-row mask words),
//              F  the up [and gate] rows, then the transposed-down rows, of
//                 its slice of the active list.
// Phases H and S read weights only, so the producer issues them as soon as
// ring slots free up -- across the grid-wide barriers between phases and
// across layers -- while the consumers still work on earlier phases; only F
// waits for the block's slice of the active list. The consumers run
//   H  hid = ReLU(W1 . x + b1) for the block's rows      -> grid barrier
//   S  s = W2 . hid + b2, one ballot per 32 slots        -> grid barrier
//   F  scan of the mask words, the block's slice, up/gate dot products, the
//      activation, h_i * downT_i into one partial sum of y per block
//                                                        -> grid barrier
//   R  the block's columns of y (partials added in a fixed order) and
//      x_{l+1} = x_l + y                                 -> grid barrier
// The grid barriers are a counter and a generation word in global memory,
// every wait bounded (a wait that runs out records SFFN_ERR_TIMEOUT and the
// kernel winds down). Every sum has the order of the per-layer kernels
// (k_pred_hidden, k_ffn, k_ffn_reduce), so hid, the FFN partials and y are
// bit-identical to sffn_decode_step's on the same masks.
#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace sffn {

namespace {

constexpr int kSW = 8;                  // consumer warps
constexpr int kSC = kSW * 32;           // consumer threads
constexpr int kSThreads = kSC + 32;     // + the producer warp
constexpr uint32_t kSB = 32768;         // ring stage bytes
constexpr int kReduceGroupsS = 32;      // partial groups of the y reduction (as k_ffn_reduce)
constexpr int kReducePer = 8;           // partials per group (blocks <= 256), zeros past the last
constexpr int kWordsPerThread = 8;      // mask words per consumer thread in the scan (f <= 65536)

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kSC) : "memory"); }

// Consumer barrier that also ORs a predicate over the 256 consumer threads:
// every consumer gets the same answer (a block-uniform abort decision).
__device__ __forceinline__ bool cbar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kSC)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

// Exclusive prefix sum of one int per consumer thread (256 threads).
__device__ __forceinline__ int cons_exclusive_scan(int v, int* s_tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(SFFN_FULL_MASK, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_tmp[warp] = x;
  cbar();
  if (warp == 0) {
    int w = lane < kSW ? s_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < kSW; o <<= 1) {
      const int y = __shfl_up_sync(SFFN_FULL_MASK, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSW) s_tmp[lane] = w;
  }
  cbar();
  const int before = warp ? s_tmp[warp - 1] : 0;
  *total = s_tmp[kSW - 1];
  cbar();
  return before + x - v;
}

struct StackLayerDev {
  const void* W1;
  const float* b1;  // null: no bias
  const void* W2;
  const float* b2;
  const void* up;
  const void* gate;
  const void* downT;
};

struct StackParams {
  const StackLayerDev* layers;
  int n_layers;
  int d, f, h, G, n_groups, nw, gwords;
  int stages;     // ring depth
  int list_cap;   // largest per-block slice of the active list
  int hr_cap;     // largest per-block share of W1 rows
  int sw_cap;     // largest per-block share of mask words
  float thres;
  const float* x0;       // input of layer 0
  float* xs;             // [n_layers][d]: x_{l+1} = x_l + y_l
  float* ys;             // [n_layers][d] or null
  uint32_t* nmask;       // [n_layers][nw]
  uint32_t* gmask;       // [n_layers][gwords] or null
  int32_t* idx;          // [n_layers][f] or null
  int32_t* count;        // [n_layers] or null
  float* hid;            // workspace [h]
  float* partials;       // workspace [grid][d]
  unsigned* bar;         // [0] arrivals, [1] generation
  uint32_t* err;
};

// Grid-wide barrier among the consumer warps of every block: an arrival
// counter and a generation word in global memory. The last block to arrive
// resets the counter and advances the generation (release); the others poll
// the generation (acquire). `ok_in` is this thread's state: if any consumer
// thread of the block has failed, the block does not arrive. Returns,
// uniformly over the block's consumers, false if the block failed, a wait ran
// out or another block failed (the reason is in the error word).
__device__ bool grid_sync(const StackParams& p, bool ok_in, unsigned* s_gen, int* s_ok) {
  if (cbar_or(!ok_in)) return false;  // every consumer thread has issued its global writes
  if (threadIdx.x == 0) {
    int ok = ld_volatile_u32(p.err) == 0;
    const unsigned gen = *s_gen;
    __threadfence();
    const unsigned old = atomicAdd(&p.bar[0], 1u);
    if (old == gridDim.x - 1) {
      atomicExch(&p.bar[0], 0u);
      __threadfence();
      st_release_u32(&p.bar[1], gen + 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u32(&p.bar[1]) == gen) {
        if (ld_volatile_u32(p.err) != 0) {
          ok = 0;
          break;
        }
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          set_device_error(p.err, SFFN_ERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    *s_gen = gen + 1u;
    *s_ok = ok;
  }
  cbar();
  return *s_ok != 0;
}

template <typename T, int ACT, int CPT>
__global__ void __launch_bounds__(kSThreads, 1) k_decode_stack(const StackParams p) {
  constexpr int EPC = WType<T>::kPerChunk;  // 8 (16-bit weights)
  constexpr bool GATED = act_gated(ACT);
  constexpr int NMAT = GATED ? 2 : 1;
  const int d = p.d, h = p.h;
  const uint32_t rowB = (uint32_t)d * 2u;      // one W1 / up / gate / downT row
  const uint32_t hrowB = (uint32_t)h * 2u;     // one W2 row
  const int nch = d / EPC;                     // 16-byte chunks of a row
  const int nchh = h / EPC;                    // 16-byte chunks of a W2 row
  const int UH = (int)(kSB / rowB);            // W1 rows per stage
  int RS = 32;                                 // W2 rows per stage: a power of two dividing 32
  while ((uint32_t)RS * hrowB > kSB) RS >>= 1;
  const int TPR = kSC / RS;                    // consumer threads per W2 row
  const int NPS = (int)(kSB / (rowB * NMAT));  // neurons per phase-A stage
  const int RPB = NPS * NMAT;                  // downT rows per phase-B stage
  const int NS = p.stages;
  const int nb = gridDim.x, b = blockIdx.x;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)NS * kSB);
  uint64_t* empty = full + NS;
  uint32_t* s_words = reinterpret_cast<uint32_t*>(empty + NS);
  int* s_off = reinterpret_cast<int*>(s_words + p.nw);
  int32_t* s_list = reinterpret_cast<int32_t*>(s_off + p.nw);
  float* s_h = reinterpret_cast<float*>(s_list + p.list_cap);
  float* s_part = s_h + p.list_cap;                        // [list_cap][8][2]
  float* s_hp = s_part + (size_t)p.list_cap * kSW * 2;     // [hr_cap][8]
  float* s_sc = s_hp + (size_t)p.hr_cap * kSW;             // [sw_cap * 32]
  __shared__ uint64_t s_ready;  // the block's slice of the active list is in s_list
  __shared__ int s_tmp[kSW];
  __shared__ int s_nloc;
  __shared__ int s_abort;
  __shared__ unsigned s_gen;
  __shared__ int s_ok;
  __shared__ float s_red[kSW][kReduceGroupsS][4];

  // block shares that do not depend on data
  const int hr0 = (int)((long long)h * b / nb), hr1 = (int)((long long)h * (b + 1) / nb);
  const int nh = hr1 - hr0;
  const int nHs = (nh + UH - 1) / UH;
  const int w0 = (int)((long long)p.nw * b / nb), w1 = (int)((long long)p.nw * (b + 1) / nb);
  const int nwl = w1 - w0;
  const int nSs = nwl * (32 / RS);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSW);
    }
    mbar_init(&s_ready, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == kSW) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      uint32_t u = 0;  // stages issued
      bool ok = true;
      // wait until stage u may be refilled
      auto acquire = [&](uint32_t uu) -> bool {
        if (*(volatile int*)&s_abort) return false;
        if (uu < (uint32_t)NS) return true;
        if (!mbar_wait_bounded(&empty[uu % NS], ((uu / NS) - 1) & 1)) {
          set_device_error(p.err, SFFN_ERR_TIMEOUT);
          return false;
        }
        return !*(volatile int*)&s_abort;
      };
      for (int l = 0; l < p.n_layers && ok; ++l) {
        const StackLayerDev Ld = p.layers[l];
        const unsigned char* W1 = static_cast<const unsigned char*>(Ld.W1);
        const unsigned char* W2 = static_cast<const unsigned char*>(Ld.W2);
        // H: W1 rows [hr0, hr1), UH per stage
        for (int k = 0; k < nHs && ok; ++k, ++u) {
          if (!(ok = acquire(u))) break;
          const int r0 = hr0 + k * UH, nr = min(UH, hr1 - r0);
          uint64_t* fb = &full[u % NS];
          mbar_arrive_expect_tx(fb, (uint32_t)nr * rowB);
          bulk_g2s(ring + (size_t)(u % NS) * kSB, W1 + (size_t)r0 * rowB, (uint32_t)nr * rowB, fb, pol);
        }
        // S: W2 rows of words [w0, w1), RS rows per stage (one contiguous copy)
        for (int k = 0; k < nSs && ok; ++k, ++u) {
          if (!(ok = acquire(u))) break;
          uint64_t* fb = &full[u % NS];
          mbar_arrive_expect_tx(fb, (uint32_t)RS * hrowB);
          bulk_g2s(ring + (size_t)(u % NS) * kSB, W2 + ((size_t)w0 * 32 + (size_t)k * RS) * hrowB,
                   (uint32_t)RS * hrowB, fb, pol);
        }
        if (!ok) break;
        // the next layer's W1 rows of this block (the first layer's for the
        // next token) into L2 while the mask is formed and scanned
        {
          const StackLayerDev& Ln = p.layers[(l + 1) % p.n_layers];
          const unsigned char* nW1 = static_cast<const unsigned char*>(Ln.W1) + (size_t)hr0 * rowB;
          const size_t bytes = (size_t)nh * rowB;
          for (size_t o = 0; o < bytes; o += 65536) prefetch_l2_bulk(nW1 + o, (uint32_t)min(bytes - o, (size_t)65536));
        }
        // F: wait for the block's slice of this layer's active list
        if (!mbar_wait_bounded(&s_ready, (uint32_t)(l & 1))) {
          set_device_error(p.err, SFFN_ERR_TIMEOUT);
          ok = false;
          break;
        }
        if (*(volatile int*)&s_abort) {
          ok = false;
          break;
        }
        const int n_local = *(volatile int*)&s_nloc;
        const int nA = (n_local + NPS - 1) / NPS, nB = (n_local + RPB - 1) / RPB;
        const unsigned char* up = static_cast<const unsigned char*>(Ld.up);
        const unsigned char* gate = static_cast<const unsigned char*>(Ld.gate);
        const unsigned char* downT = static_cast<const unsigned char*>(Ld.downT);
        for (int v = 0; v < nA && ok; ++v, ++u) {
          if (!(ok = acquire(u))) break;
          const int k0 = v * NPS, nk = min(NPS, n_local - k0);
          uint64_t* fb = &full[u % NS];
          unsigned char* dst = ring + (size_t)(u % NS) * kSB;
          mbar_arrive_expect_tx(fb, (uint32_t)nk * NMAT * rowB);
          for (int k = 0; k < nk; ++k) {
            const size_t slot = (size_t)s_list[k0 + k];
            unsigned char* dk = dst + (size_t)k * NMAT * rowB;
            bulk_g2s(dk, up + slot * rowB, rowB, fb, pol);
            if (GATED) bulk_g2s(dk + rowB, gate + slot * rowB, rowB, fb, pol);
          }
        }
        for (int v = 0; v < nB && ok; ++v, ++u) {
          if (!(ok = acquire(u))) break;
          const int r0 = v * RPB, nr = min(RPB, n_local - r0);
          uint64_t* fb = &full[u % NS];
          unsigned char* dst = ring + (size_t)(u % NS) * kSB;
          mbar_arrive_expect_tx(fb, (uint32_t)nr * rowB);
          for (int i = 0; i < nr; ++i)
            bulk_g2s(dst + (size_t)i * rowB, downT + (size_t)s_list[r0 + i] * rowB, rowB, fb, pol);
        }
      }
      if (!ok) {
        atomicExch(&s_abort, 1);
        // let the copies that may still be in flight land
        for (uint32_t q = u > (uint32_t)NS ? u - NS : 0; q < u; ++q)
          mbar_wait_bounded(&full[q % NS], (q / NS) & 1);
      }
    }
  } else {
    // ================================================================ consumers
    pdl_launch_dependents();
    pdl_wait();  // x0 may come from the previous kernel
    if (threadIdx.x == 0) s_gen = ld_acquire_u32(&p.bar[1]);
    cbar();
    uint32_t u = 0;  // stages consumed
    bool ok = true;
    // wait for stage u's bytes; false if a wait ran out or the block aborts
    // (a warp that fails leaves its stage loop; the block decides uniformly
    // at the next cbar_or / grid_sync)
    auto wait_full = [&](uint32_t uu) -> bool {
      const bool got = __all_sync(SFFN_FULL_MASK, mbar_wait_bounded(&full[uu % NS], (uu / NS) & 1));
      if (!got || __any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
        if (!got && lane == 0) set_device_error(p.err, SFFN_ERR_TIMEOUT);
        if (lane == 0) atomicExch(&s_abort, 1);
        return false;
      }
      return true;
    };
    auto release = [&](uint32_t uu) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[uu % NS]);
    };
    for (int l = 0; l < p.n_layers; ++l) {
      const StackLayerDev Ld = p.layers[l];
      const float* x = l == 0 ? p.x0 : p.xs + (size_t)(l - 1) * d;
      // ---------------------------------------------------------- H
      {
        float xr[CPT][EPC];
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int c = threadIdx.x + j * kSC;
#pragma unroll
          for (int e = 0; e < EPC; e += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < nch) v = ld_dep4(x + (size_t)c * EPC + e);
            xr[j][e] = v.x; xr[j][e + 1] = v.y; xr[j][e + 2] = v.z; xr[j][e + 3] = v.w;
          }
        }
        for (int k = 0; k < nHs; ++k, ++u) {
          if (!(ok = ok && wait_full(u))) break;
          const int nr = min(UH, nh - k * UH);
          const unsigned char* sp = ring + (size_t)(u % NS) * kSB;
          for (int r = 0; r < nr; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
              const int c = threadIdx.x + j * kSC;
              if (c < nch) acc += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + (size_t)r * rowB + (size_t)c * 16), xr[j]);
            }
            acc = warp_sum(acc);
            if (lane == 0) s_hp[(k * UH + r) * kSW + warp] = acc;
          }
          release(u);
        }
        if (cbar_or(!ok)) {
          ok = false;
          break;
        }
        if ((int)threadIdx.x < nh) {
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kSW; ++w) s += s_hp[threadIdx.x * kSW + w];
          if (Ld.b1) s += Ld.b1[hr0 + threadIdx.x];
          __stcg(p.hid + hr0 + threadIdx.x, relu_nan(s));
        }
      }
      if (!(ok = grid_sync(p, ok, &s_gen, &s_ok))) break;
      // ---------------------------------------------------------- S
      {
        const int r = threadIdx.x / TPR, q = threadIdx.x % TPR;
        float hv[8][EPC];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = q + k * TPR;
#pragma unroll
          for (int e = 0; e < EPC; e += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < nchh) v = ld_dep4(p.hid + (size_t)c * EPC + e);
            hv[k][e] = v.x; hv[k][e + 1] = v.y; hv[k][e + 2] = v.z; hv[k][e + 3] = v.w;
          }
        }
        for (int k = 0; k < nSs; ++k, ++u) {
          if (!(ok = ok && wait_full(u))) break;
          const unsigned char* sp = ring + (size_t)(u % NS) * kSB + (size_t)r * hrowB;
          float acc = 0.f;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int c = q + kk * TPR;
            if (c < nchh) acc += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + (size_t)c * 16), hv[kk]);
          }
          for (int o = TPR >> 1; o >= 1; o >>= 1) acc += __shfl_xor_sync(SFFN_FULL_MASK, acc, o);
          if (q == 0) {
            const int row = k * RS + r;  // within the block's rows
            if (Ld.b2) acc += Ld.b2[(size_t)w0 * 32 + row];
            s_sc[row] = acc;
          }
          release(u);
        }
        if (cbar_or(!ok)) {
          ok = false;
          break;
        }
        {
          uint32_t* nm = p.nmask + (size_t)l * p.nw;
          for (int k = warp; k < nwl; k += kSW) {
            const uint32_t m = __ballot_sync(SFFN_FULL_MASK, s_sc[k * 32 + lane] >= p.thres);  // NaN: inactive
            if (lane == 0) __stcg(nm + w0 + k, m);
          }
        }
      }
      if (!(ok = grid_sync(p, ok, &s_gen, &s_ok))) break;
      // ---------------------------------------------------------- F
      const uint32_t* nm = p.nmask + (size_t)l * p.nw;
      int total, lo, n_local;
      {
        // all words requested at once (coalesced, independent loads), then
        // each thread counts a contiguous range of them
        uint32_t wv[kWordsPerThread];
#pragma unroll
        for (int i = 0; i < kWordsPerThread; ++i) {
          const int w = threadIdx.x + i * kSC;
          wv[i] = w < p.nw ? __ldcg(nm + w) : 0u;
        }
#pragma unroll
        for (int i = 0; i < kWordsPerThread; ++i) {
          const int w = threadIdx.x + i * kSC;
          if (w < p.nw) s_words[w] = wv[i];
        }
        cbar();
        const int per = (p.nw + kSC - 1) / kSC;
        const int a0 = min(p.nw, (int)threadIdx.x * per), a1 = min(p.nw, a0 + per);
        int cnt = 0;
        for (int w = a0; w < a1; ++w) cnt += __popc(s_words[w]);
        int off = cons_exclusive_scan(cnt, s_tmp, &total);
        for (int w = a0; w < a1; ++w) {
          s_off[w] = off;
          off += __popc(s_words[w]);
        }
        cbar();
        lo = (int)((long long)total * b / nb);
        const int hi = (int)((long long)total * (b + 1) / nb);
        n_local = min(hi - lo, p.list_cap);
        for (int w = threadIdx.x; w < p.nw; w += kSC) {
          uint32_t m = s_words[w];
          int pos = s_off[w];
          if (pos >= lo + n_local || pos + __popc(m) <= lo) continue;
          while (m) {
            const int bit = __ffs(m) - 1;
            m &= m - 1;
            if (pos >= lo && pos < lo + n_local) s_list[pos - lo] = w * 32 + bit;
            ++pos;
          }
        }
        if (b == 0) {
          if (threadIdx.x == 0 && p.count) p.count[l] = total;
          if (p.gmask) {
            const int wpg = p.G / 32;
            uint32_t* gm = p.gmask + (size_t)l * p.gwords;
            for (int g = threadIdx.x; g < p.gwords * 32; g += kSC) {
              bool a = false;
              if (g < p.n_groups)
                for (int k = 0; k < wpg; ++k) a |= (s_words[g * wpg + k] != 0u);
              const uint32_t word = __ballot_sync(SFFN_FULL_MASK, a);
              if (lane == 0) gm[g >> 5] = word;
            }
          }
        }
        cbar();
        if (threadIdx.x == 0) {
          s_nloc = n_local;
          mbar_arrive(&s_ready);  // release: s_list and s_nloc to the producer
        }
      }
      const int nA = (n_local + NPS - 1) / NPS, nB = (n_local + RPB - 1) / RPB;
      {
        float xr[CPT][EPC];
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int c = threadIdx.x + j * kSC;
#pragma unroll
          for (int e = 0; e < EPC; e += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < nch) v = ld_dep4(x + (size_t)c * EPC + e);
            xr[j][e] = v.x; xr[j][e + 1] = v.y; xr[j][e + 2] = v.z; xr[j][e + 3] = v.w;
          }
        }
        for (int v = 0; v < nA; ++v, ++u) {
          if (!(ok = ok && wait_full(u))) break;
          const int k0 = v * NPS;
          const unsigned char* sp0 = ring + (size_t)(u % NS) * kSB;
          for (int k = 0; k < NPS; ++k) {
            if (k0 + k >= n_local) break;
            const unsigned char* sp = sp0 + (size_t)k * NMAT * rowB;
            float pu = 0.f, pg = 0.f;
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
              const int c = threadIdx.x + j * kSC;
              if (c < nch) {
                pu += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + (size_t)c * 16), xr[j]);
                if (GATED) pg += dot_chunk<T>(*reinterpret_cast<const uint4*>(sp + rowB + (size_t)c * 16), xr[j]);
              }
            }
            pu = warp_sum(pu);
            if (GATED) pg = warp_sum(pg);
            if (lane == 0) {
              s_part[((size_t)(k0 + k) * kSW + warp) * 2] = pu;
              s_part[((size_t)(k0 + k) * kSW + warp) * 2 + 1] = pg;
            }
          }
          release(u);
        }
      }
      if (cbar_or(!ok)) {
          ok = false;
          break;
        }
      {
        int32_t* idx_out = p.idx ? p.idx + (size_t)l * p.f : nullptr;
        for (int a = threadIdx.x; a < n_local; a += kSC) {
          float uu = 0.f, gg = 0.f;
#pragma unroll
          for (int w = 0; w < kSW; ++w) {
            uu += s_part[((size_t)a * kSW + w) * 2];
            gg += s_part[((size_t)a * kSW + w) * 2 + 1];
          }
          s_h[a] = neuron_act<ACT>(uu, gg);
          if (idx_out) idx_out[lo + a] = s_list[a];
        }
      }
      cbar();
      {
        float acc[CPT][EPC];
#pragma unroll
        for (int j = 0; j < CPT; ++j)
#pragma unroll
          for (int e = 0; e < EPC; ++e) acc[j][e] = 0.f;
        for (int v = 0; v < nB; ++v, ++u) {
          if (!(ok = ok && wait_full(u))) break;
          const unsigned char* sp = ring + (size_t)(u % NS) * kSB;
          const int r0 = v * RPB, nr = min(RPB, n_local - r0);
          for (int i = 0; i < nr; ++i) {
            const float hvv = s_h[r0 + i];
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
              const int c = threadIdx.x + j * kSC;
              if (c < nch) {
                float w[EPC];
                WType<T>::unpack(*reinterpret_cast<const uint4*>(sp + (size_t)i * rowB + (size_t)c * 16), w);
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[j][e] = fmaf(hvv, w[e], acc[j][e]);
              }
            }
          }
          release(u);
        }
        float* part = p.partials + (size_t)b * d;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int c = threadIdx.x + j * kSC;
          if (c < nch) {
#pragma unroll
            for (int e = 0; e < EPC; e += 4)
              __stcg(reinterpret_cast<float4*>(part + (size_t)c * EPC + e),
                     make_float4(acc[j][e], acc[j][e + 1], acc[j][e + 2], acc[j][e + 3]));
          }
        }
      }
      if (!(ok = grid_sync(p, ok, &s_gen, &s_ok))) break;
      // ---------------------------------------------------------- R
      {
        // float4 columns [c0, c1) of this block; for each column lane g of a
        // warp adds partials g, g + 32, ... and the 32 group sums are added in
        // group order (the order of k_ffn_reduce)
        const int cols = d / 4;
        const int c0 = (int)((long long)cols * b / nb), c1 = (int)((long long)cols * (b + 1) / nb);
        float* yl = p.ys ? p.ys + (size_t)l * d : nullptr;
        float* xo = p.xs + (size_t)l * d;
        // two columns per warp and pass, every partial load issued before any add
        for (int cb = c0 + warp; cb < c1; cb += 2 * kSW) {
          float4 v[2][kReducePer];
          float xv[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c = cb + k * kSW;
            xv[k] = (lane < 4 && c < c1) ? ld_dep(x + (size_t)c * 4 + lane) : 0.f;
#pragma unroll
            for (int i = 0; i < kReducePer; ++i) {
              const int pi = lane + i * kReduceGroupsS;
              v[k][i] = (c < c1 && pi < nb) ? ld_dep4(p.partials + (size_t)pi * d + (size_t)c * 4)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c = cb + k * kSW;
            float4 acc = v[k][0];
#pragma unroll
            for (int i = 1; i < kReducePer; ++i) {
              acc.x += v[k][i].x; acc.y += v[k][i].y; acc.z += v[k][i].z; acc.w += v[k][i].w;
            }
            s_red[warp][lane][0] = acc.x;
            s_red[warp][lane][1] = acc.y;
            s_red[warp][lane][2] = acc.z;
            s_red[warp][lane][3] = acc.w;
            __syncwarp();
            if (lane < 4 && c < c1) {
              float sum = s_red[warp][0][lane];
              for (int g = 1; g < kReduceGroupsS; ++g) sum += s_red[warp][g][lane];
              if (yl) yl[(size_t)c * 4 + lane] = sum;
              __stcg(xo + (size_t)c * 4 + lane, xv[k] + sum);
            }
            __syncwarp();
          }
        }
      }
      if (l + 1 < p.n_layers && !(ok = grid_sync(p, ok, &s_gen, &s_ok))) break;
    }
    if (threadIdx.x == 0 && !ok) atomicExch(&s_abort, 1);
  }
  __syncthreads();
}

}  // namespace

// ------------------------------------------------------------------ host side

struct StackShape {
  int stages = 0, list_cap = 0, hr_cap = 0, sw_cap = 0;
  size_t smem = 0;
};

static StackShape stack_shape(const sffn_layer& L, int nb, int smem_optin) {
  StackShape s;
  const int f = L.desc.f, h = L.desc.h, nw = L.nwords;
  s.list_cap = (f + nb - 1) / nb + 1;
  s.hr_cap = (h + nb - 1) / nb;
  s.sw_cap = (nw + nb - 1) / nb;
  const size_t fixed = (size_t)nw * 8 + (size_t)s.list_cap * (4 + 4 + kSW * 2 * 4) + (size_t)s.hr_cap * kSW * 4 +
                       (size_t)s.sw_cap * 32 * 4;
  const size_t stat = sizeof(float) * kSW * kReduceGroupsS * 4 + 256;  // static shared memory and slack
  const size_t avail = (size_t)smem_optin > fixed + stat ? (size_t)smem_optin - fixed - stat : 0;
  s.stages = (int)std::min<size_t>(8, avail / (kSB + 16));
  s.smem = (size_t)s.stages * (kSB + 16) + fixed;
  return s;
}

bool stack_supported(const sffn_layer& L, std::string* why) {
  const sffn_layer_desc& D = L.desc;
  if (D.ffn_format != SFFN_FFN_ROWS) {
    *why = "the stack kernel reads 16-bit FFN rows (8-bit and 4-bit rows: use the per-layer calls)";
    return false;
  }
  if (D.wdtype == SFFN_F32) {
    *why = "the stack kernel needs 16-bit weights (fp16 or bf16)";
    return false;
  }
  const size_t rowB = (size_t)D.d * 2;
  if (rowB * (act_gated(D.act) ? 2 : 1) > kSB) {
    *why = "one neuron's up/gate rows must fit a 32 KB ring stage (d <= 8192 gated, d <= 16384 otherwise)";
    return false;
  }
  if (L.num_sms > kReduceGroupsS * kReducePer) {
    *why = "the stack kernel's reduction handles at most 256 SMs";
    return false;
  }
  StackShape s = stack_shape(L, L.num_sms, L.smem_optin);
  if (s.stages < 3) {
    *why = "the stack kernel's ring does not fit in shared memory for this shape";
    return false;
  }
  return true;
}

namespace {

template <typename T, int ACT>
cudaError_t set_stack_attr_t(int smem) {
  cudaError_t e;
  if ((e = set_dynamic_smem_max(k_decode_stack<T, ACT, 1>, smem))) return e;
  if ((e = set_dynamic_smem_max(k_decode_stack<T, ACT, 2>, smem))) return e;
  if ((e = set_dynamic_smem_max(k_decode_stack<T, ACT, 4>, smem))) return e;
  return set_dynamic_smem_max(k_decode_stack<T, ACT, 8>, smem);
}

template <typename T>
cudaError_t set_stack_attr(int smem) {
  cudaError_t e;
  if ((e = set_stack_attr_t<T, SFFN_ACT_RELU>(smem))) return e;
  if ((e = set_stack_attr_t<T, SFFN_ACT_REGLU>(smem))) return e;
  if ((e = set_stack_attr_t<T, SFFN_ACT_SWIGLU>(smem))) return e;
  return set_stack_attr_t<T, SFFN_ACT_RELU2>(smem);
}

template <typename T, int ACT>
cudaError_t launch_stack_t(int cpt, dim3 grid, size_t smem, cudaStream_t st, const StackParams& p) {
  switch (cpt) {
    case 1: return launch_ex(k_decode_stack<T, ACT, 1>, grid, dim3(kSThreads), smem, st, true, 1, p);
    case 2: return launch_ex(k_decode_stack<T, ACT, 2>, grid, dim3(kSThreads), smem, st, true, 1, p);
    case 4: return launch_ex(k_decode_stack<T, ACT, 4>, grid, dim3(kSThreads), smem, st, true, 1, p);
    default: return launch_ex(k_decode_stack<T, ACT, 8>, grid, dim3(kSThreads), smem, st, true, 1, p);
  }
}

template <typename T>
cudaError_t launch_stack_act(int act, int cpt, dim3 grid, size_t smem, cudaStream_t st, const StackParams& p) {
  switch (act) {
    case SFFN_ACT_RELU: return launch_stack_t<T, SFFN_ACT_RELU>(cpt, grid, smem, st, p);
    case SFFN_ACT_REGLU: return launch_stack_t<T, SFFN_ACT_REGLU>(cpt, grid, smem, st, p);
    case SFFN_ACT_RELU2: return launch_stack_t<T, SFFN_ACT_RELU2>(cpt, grid, smem, st, p);
    default: return launch_stack_t<T, SFFN_ACT_SWIGLU>(cpt, grid, smem, st, p);
  }
}

}  // namespace

cudaError_t configure_stack_kernels(const sffn_layer& L) {
  return L.desc.wdtype == SFFN_F16 ? set_stack_attr<__half>(L.smem_optin) : set_stack_attr<__nv_bfloat16>(L.smem_optin);
}

size_t stack_ws_bytes(const sffn_layer& L) {
  const size_t hid = ((size_t)L.desc.h * 4 + 255) & ~size_t(255);
  return hid + (size_t)L.num_sms * L.desc.d * 4;
}

cudaError_t launch_stack(const sffn_stack& S, const float* x0, float* xs, float* ys, float thres,
                         const sffn_masks& m, void* ws, cudaStream_t st) {
  const sffn_layer& L = *S.layers[0];
  const int nb = L.num_sms;
  StackShape sh = stack_shape(L, nb, L.smem_optin);
  StackParams p = {};
  p.layers = static_cast<const StackLayerDev*>(S.dev_layers);
  p.n_layers = S.n_layers;
  p.d = L.desc.d;
  p.f = L.desc.f;
  p.h = L.desc.h;
  p.G = L.desc.group_size;
  p.n_groups = L.n_groups;
  p.nw = L.nwords;
  p.gwords = L.gwords;
  p.stages = sh.stages;
  p.list_cap = sh.list_cap;
  p.hr_cap = sh.hr_cap;
  p.sw_cap = sh.sw_cap;
  p.thres = thres;
  p.x0 = x0;
  p.xs = xs;
  p.ys = ys;
  p.nmask = m.nmask;
  p.gmask = m.gmask;
  p.idx = m.idx;
  p.count = m.count;
  char* base = static_cast<char*>(ws);
  p.hid = reinterpret_cast<float*>(base);
  p.partials = reinterpret_cast<float*>(base + (((size_t)L.desc.h * 4 + 255) & ~size_t(255)));
  p.bar = S.bar;
  p.err = S.err;
  const int nch = L.desc.d / 8;
  const int need = (nch + kSC - 1) / kSC;
  const int cpt = need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
  if (L.desc.wdtype == SFFN_F16) return launch_stack_act<__half>(L.desc.act, cpt, dim3(nb), sh.smem, st, p);
  return launch_stack_act<__nv_bfloat16>(L.desc.act, cpt, dim3(nb), sh.smem, st, p);
}

size_t stack_layer_desc_bytes() { return sizeof(StackLayerDev); }

void stack_fill_layer_desc(const sffn_layer& L, void* out) {
  StackLayerDev d;
  d.W1 = L.W1;
  d.b1 = L.has_b1 ? L.b1 : nullptr;
  d.W2 = L.W2;
  d.b2 = L.has_b2 ? L.b2 : nullptr;
  d.up = L.up;
  d.gate = L.gate;
  d.downT = L.downT;
  *static_cast<StackLayerDev*>(out) = d;
}

}  // namespace sffn
