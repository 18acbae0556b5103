// Batched decode (B > 1): the union of the batch's predicted masks decides
// which FFN rows are read, each token keeps its own mask for its own output
// (KAIROX 问题与动机: larger batches raise the number of activated neurons;
// PowerInfer §5.3-§5.4 neuron-aware operators). Every contraction of a batch
// step is a tall-skinny product (many weight rows, N = 16 or 32 tokens) run
// on the fifth-generation tensor cores:
//   hidden  D[h x N]  = W1 [contiguous rows, K = d]          . X^T
//   scores  D[f x N]  = W2 [contiguous rows, K = h]          . HID^T
//   up/gate D[U x N]  = up, gate [union rows, K = d]         . X^T
//   down    D[d x N]  = downT^T [K = union rows, MN-major A] . H^T
// by one persistent kernel (k_tc_gemm) that writes fp32 partial products
// over K splits; small CUDA-core kernels finish each step (bias, ReLU,
// threshold + ballot, activation with the per-token mask, residual).
// Activations enter the tensor cores as a high and a low 16-bit part
// (v = hi + lo, two MMAs accumulating into the same fp32 tile), which keeps
// their product with the 16-bit weights close to fp32 accuracy.
#include "common.cuh"
#include "internal.h"
#include "scan.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <string>

namespace sffn {

namespace {

constexpr int kGemmThreads = 256;    // warps 0-3 producers, warp 4 MMA issuer, warps 4-7 epilogue
constexpr int kProducers = 128;
constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr int kGemmSmemBudget = 221 * 1024;
constexpr int kViewThreadsB = 1024;

struct GemmArgs {
  CUtensorMap tmA;          // contiguous A rows (products without a row list): box 64 K x 128 rows
  CUtensorMap tmB;          // B parts [2 * npad][ldb]: box 64 K x npad rows
  const unsigned char* A0;  // first A matrix
  const unsigned char* A1;  // second A matrix with the same rows (gate), or null
  const int32_t* rows;      // gathered rows of A (null: row i is row i)
  const int32_t* count_dev; // device extent of the row-indexed dimension (null: fixed_count)
  int fixed_count;
  int other;                // K-major: K extent; MN-major: M extent (elements, multiple of 64 / 128)
  int lda;                  // elements per A row
  const unsigned char* Bhl; // [2][npad][ldb] 16-bit hi then lo parts, K-major
  int ldb;
  float* D;                 // partial tiles [slot][npad][tile rows] (slot = CTA + tile, see Plan)
  size_t dmat_stride;       // floats from the first matrix's partials to the second's
  int grid;                 // CTAs launched
  uint32_t* err;
};

// Work decomposition shared by the GEMM and its finishers (stream-K): the
// m_tiles x kblocks (tile, K step) pairs, tile after tile, are cut into
// `ctas` equal contiguous ranges, one per CTA, so every CTA streams the same
// number of ring stages. A CTA writes one partial tile for every tile its
// range touches, at slot CTA + tile (unique: a later CTA starts where the
// earlier one ends); the CTAs touching tile t are cta_of(t * kblocks) ..
// cta_of((t + 1) * kblocks - 1), whose partials the finishers add in CTA
// order. A K step is `ksub` blocks of 64 (K-major products); an MN-major tile
// is `msub` blocks of 128 output rows.
struct Plan {
  int m_tiles, kblocks, ctas, tile_rows;
  long long total;
};

__host__ __device__ inline Plan make_plan(bool mn_major, int count, int other, int grid, int ksub = 1,
                                          int msub = 1) {
  Plan p;
  if (!mn_major) {
    p.tile_rows = kTileM;
    p.m_tiles = (count + kTileM - 1) / kTileM;
    p.kblocks = other / (kTileK * ksub);
  } else {
    p.tile_rows = kTileM * msub;
    p.m_tiles = other / p.tile_rows;
    p.kblocks = (count + kTileK - 1) / kTileK;
  }
  p.total = (long long)p.m_tiles * p.kblocks;
  p.ctas = (int)(p.total < grid ? p.total : grid);
  return p;
}

// Ring-stage shapes. Each stage reads longer contiguous runs of every weight
// row than one 128-byte K block: HBM serves such runs much faster than
// scattered 128-byte pieces.
//   contiguous rows (TMA): 4 K blocks (512 bytes per row) when K allows;
__host__ __device__ inline int ksub_contig(int k) { return k % (4 * kTileK) == 0 ? 4 : 1; }
//   gathered K-major rows (cp.async): 2 K blocks (256 bytes per row), which
//   leaves room for four stages (measured faster than 4 K blocks in two);
__host__ __device__ inline int ksub_gather(int k, int nmat) {
  (void)nmat;
  return k % (2 * kTileK) == 0 ? 2 : 1;
}
//   gathered MN-major rows (down): 4 output tiles of 128 (1 KB per row) when d allows.
__host__ __device__ inline int msub_down(int d) {
  const int t = d / kTileM;
  return t % 4 == 0 ? 4 : (t % 2 == 0 ? 2 : 1);
}

__host__ __device__ inline bool cta_in_plan(const Plan& p, int b) { return b < p.ctas; }

// First linear (tile, K step) index of CTA b's range.
__host__ __device__ inline long long range_lo(const Plan& p, int b) { return p.total * b / p.ctas; }

// The CTA whose range holds linear index x (p.total > 0).
__host__ __device__ inline int cta_of(const Plan& p, long long x) {
  return (int)(((x + 1) * p.ctas - 1) / p.total);
}

// One persistent kernel per product. A tiles come from the TMA engine when the
// rows are contiguous (GATHER false: the hidden and scores products) or from
// coalesced cp.async copies of the gathered union rows (GATHER true); the B
// tile of each K block (the activations' hi parts in rows 0..NPAD-1 and lo
// parts in rows NPAD..2*NPAD-1) always comes from the TMA engine, so one MMA
// of N = 2 * NPAD covers both parts and the epilogue adds the two halves.
// Per ring stage, `tfull` counts the TMA bytes and `full` the 128 producer
// threads' cp.async arrivals (GATHER only); the MMA thread waits for both.
// Stage layout (every tile 1024-byte aligned): A tiles, then KSUB B tiles.
//   K-major: A tiles [KSUB][NMAT] of 128 rows x 64 K.
//   MN-major: A tiles [MSUB] of 128 M x 64 K (KSUB = 1, NMAT = 1).
template <bool MN, int NMAT, int NPAD, bool GATHER, int KSUB, int MSUB>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_tc_gemm(const __grid_constant__ GemmArgs g, bool bf16, int stages) {
  static_assert(!MN || (GATHER && KSUB == 1 && NMAT == 1), "the MN-major product gathers one K block per stage");
  static_assert(MN || MSUB == 1, "output sub-tiles belong to the MN-major product");
  static_assert(GATHER || NMAT == 1, "contiguous products have one A matrix");
  constexpr int N2 = 2 * NPAD;                    // MMA N: hi rows then lo rows of B
  constexpr uint32_t kA = kTileM * kTileK * 2;    // 16 KB per A tile
  constexpr uint32_t kBt = N2 * kTileK * 2;       // B tile of one K block
  constexpr int NACC = MN ? MSUB : NMAT;          // accumulators in tensor memory
  constexpr uint32_t kATiles = MN ? MSUB : KSUB * NMAT;
  constexpr uint32_t kStage = kATiles * kA + KSUB * kBt;
  constexpr uint32_t kCols = NACC * N2 <= 32 ? 32u : (NACC * N2 <= 64 ? 64u : (NACC * N2 <= 128 ? 128u : 256u));
  // gathered K-major rows: TPR threads per row cover its KSUB * 128 bytes
  constexpr int TPR = KSUB * 8, RPI = kProducers / TPR, NIK = kTileM / RPI;
  // gathered MN-major rows: TPK threads per K row cover its MSUB * 256 bytes
  constexpr int TPK = MSUB * 16, RPK = kProducers / TPK, NIM = kTileK / RPK;
  static_assert(!MN || NIM <= (TPK >= 32 ? 32 : 16), "row indices of a stage must fit one lane each");

  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)stages * kStage);
  uint64_t* tfull = full + stages;
  uint64_t* empty = tfull + stages;
  uint64_t* dfull = empty + stages;
  uint64_t* dempty = dfull + 1;
  uint64_t* drain = dempty + 1;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], kProducers);
      mbar_init(&tfull[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(dfull, 1);
    mbar_init(dempty, 4);
    mbar_init(drain, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 4) tc::alloc(&s_tmem, kCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = s_tmem;

  pdl_launch_dependents();
  // Contiguous products: the weights are not written by earlier kernels, so
  // thread 0 requests the A tiles of this CTA's first ring stages before the
  // wait; their B tiles (written by the previous kernel) follow after it. The
  // stage's barrier is told the bytes of both at once.
  int pre = 0;
  if (!GATHER && tid == 0) {
    const Plan p0 = make_plan(false, g.fixed_count, g.other, g.grid, KSUB, 1);
    if (cta_in_plan(p0, blockIdx.x)) {
      const uint64_t pol_a = l2_policy_evict_first();
      const long long i_lo = range_lo(p0, blockIdx.x), i_hi = range_lo(p0, blockIdx.x + 1);
      for (; pre < stages && i_lo + pre < i_hi; ++pre) {
        const long long i = i_lo + pre;
        const int mt = (int)(i / p0.kblocks), kb = (int)(i % p0.kblocks);
        unsigned char* st = ring + (size_t)pre * kStage;
        mbar_arrive_expect_tx(&tfull[pre], KSUB * (kA + kBt));
#pragma unroll
        for (int j = 0; j < KSUB; ++j)
          tc::tma_load_2d(st + j * kA, &g.tmA, (kb * KSUB + j) * kTileK, mt * kTileM, &tfull[pre], pol_a);
      }
    }
  }
  pdl_wait();  // operands and row lists come from earlier kernels
  const int count = g.count_dev ? ld_dep(g.count_dev) : g.fixed_count;
  const Plan p = make_plan(MN, count, g.other, g.grid, KSUB, MSUB);
  const int cta = blockIdx.x;
  const long long r_lo = cta < p.ctas ? range_lo(p, cta) : 0;
  const long long r_hi = cta < p.ctas ? range_lo(p, cta + 1) : 0;
  // segment [i0, i1) of this CTA's range inside tile mt, K steps [kb0, kb1)
  auto segment = [&](long long i0, int& mt, int& kb0, int& kb1, long long& i1) {
    mt = (int)(i0 / p.kblocks);
    const long long tile_end = (long long)(mt + 1) * p.kblocks;
    i1 = r_hi < tile_end ? r_hi : tile_end;
    kb0 = (int)(i0 - (long long)mt * p.kblocks);
    kb1 = (int)(i1 - (long long)mt * p.kblocks);
  };

  if (warp < 4 && (GATHER || tid == 0)) {
    // ------------------------------------------------------------ producers
    // K-major gathered rows: thread t copies 16-byte chunk t % TPR of rows
    // t / TPR + RPI * i, so a warp instruction reads whole 128-byte lines.
    // MN-major: thread t copies chunk t % TPK of K rows t / TPK + RPK * i;
    // the rows of the next stage are held one per lane (lane l: K row
    // k0 + RPK * l, k0 = t / TPK; with 16 threads per K row each half-warp
    // holds its own) and handed out by shuffles. Thread 0 issues the TMA loads.
    const uint64_t pol_a = l2_policy_evict_first();     // weights: read once per step
    const uint64_t pol_b = tc::l2_policy_evict_last();  // activations: read by every CTA
    const int k0 = tid / TPK;
    const int hbase = TPK >= 32 ? 0 : (lane & 16), li = TPK >= 32 ? lane : (lane & 15);
    int it = 0;
    for (long long i0 = r_lo, i1 = 0; i0 < r_hi; i0 = i1) {
      int mt, kb0, kb1;
      segment(i0, mt, kb0, kb1, i1);
      size_t roff[GATHER && !MN ? NIK : 1];
      if (GATHER && !MN) {
#pragma unroll
        for (int i = 0; i < NIK; ++i) {
          const int m = mt * kTileM + tid / TPR + RPI * i;
          const int r = m < count ? ld_dep(g.rows + m) : 0;
          roff[i] = (size_t)r * g.lda * 2 + (size_t)(tid % TPR) * 16;
        }
      }
      int nidx = 0;  // MN-major: this lane's row of the next stage
      if (GATHER && MN && li < NIM) {
        const int kidx = kb0 * kTileK + k0 + RPK * li;
        nidx = ld_dep(g.rows + (kidx < count ? kidx : count - 1));
      }
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % stages;
        bool ok = it < stages || mbar_wait_bounded(&empty[s], (uint32_t)((it / stages - 1) & 1));
        if (GATHER) ok = __all_sync(SFFN_FULL_MASK, ok);
        const bool stop = GATHER ? __any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)
                                 : (*(volatile int*)&s_abort != 0);
        if (!ok || stop) {
          if (!ok && lane == 0) {
            set_device_error(g.err, SFFN_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          goto producers_done;
        }
        unsigned char* st = ring + (size_t)s * kStage;
        unsigned char* sb = st + kATiles * kA;
        if (tid == 0) {
          const bool early = it < pre;  // A tiles already requested before the wait
          if (!early) mbar_arrive_expect_tx(&tfull[s], KSUB * ((GATHER ? 0u : kA) + kBt));
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
            const int kx = (kb * KSUB + j) * kTileK;
            if (!GATHER && !early) tc::tma_load_2d(st + j * kA, &g.tmA, kx, mt * kTileM, &tfull[s], pol_a);
            tc::tma_load_2d(sb + j * kBt, &g.tmB, kx, 0, &tfull[s], pol_b);
          }
        }
        if (GATHER) {
          if (!MN) {
            const int c = tid % TPR, jb = c >> 3, cj = c & 7;
            const size_t kofs = (size_t)kb * KSUB * kTileK * 2;
#pragma unroll
            for (int i = 0; i < NIK; ++i) {
              const uint32_t so = (uint32_t)(jb * NMAT) * kA + tc::kmajor_off(tid / TPR + RPI * i, cj);
              tc::cp_async16(st + so, g.A0 + roff[i] + kofs, pol_a);
              if (NMAT == 2) tc::cp_async16(st + so + kA, g.A1 + roff[i] + kofs, pol_a);
            }
          } else {
            const int cur = nidx;
            if (kb + 1 < kb1 && li < NIM) {  // the next stage's rows, loaded while this one streams
              const int kidx = (kb + 1) * kTileK + k0 + RPK * li;
              nidx = ld_dep(g.rows + (kidx < count ? kidx : count - 1));
            }
            const int c = tid % TPK, mi = c >> 4, c16 = c & 15;
            const size_t mofs = ((size_t)mt * MSUB * kTileM + (size_t)mi * kTileM + c16 * 8) * 2;
#pragma unroll
            for (int i = 0; i < NIM; ++i) {
              const int r = __shfl_sync(SFFN_FULL_MASK, cur, hbase | i);
              tc::cp_async16(st + mi * kA + tc::mnmajor_off(k0 + RPK * i, c16), g.A0 + (size_t)r * g.lda * 2 + mofs,
                             pol_a);
            }
          }
          tc::cp_async_arrive(&full[s]);
        }
      }
    }
  producers_done:
    if (GATHER) tc::cp_async_wait_all();
    // let this CTA's TMA loads that no MMA consumed land before exiting
    if (tid == 0 && *(volatile int*)&s_abort) {
      const int n = it > pre ? it : pre;
      for (int q = n > stages ? n - stages : 0; q < n; ++q)
        mbar_wait_bounded(&tfull[q % stages], (uint32_t)((q / stages) & 1));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------- MMA issue + epilogue
    const uint32_t idesc = tc::instr_desc(bf16, MN, N2);
    const int ew = warp - 4;  // TMEM lane quarter of this warp
    int it = 0, ui = 0;
    bool issued = false;
    for (long long i0 = r_lo, i1 = 0; i0 < r_hi; i0 = i1, ++ui) {
      int mt, kb0, kb1;
      segment(i0, mt, kb0, kb1, i1);
      if (warp == 4 && lane == 0) {
        bool ok = ui == 0 || mbar_wait_bounded(dempty, (uint32_t)((ui - 1) & 1));
        if (ok) tc::fence_after();
        for (int kb = kb0; ok && kb < kb1; ++kb, ++it) {
          const int s = it % stages;
          ok = mbar_wait_bounded(&tfull[s], (uint32_t)((it / stages) & 1));
          if (ok && GATHER) ok = mbar_wait_bounded(&full[s], (uint32_t)((it / stages) & 1));
          if (!ok || *(volatile int*)&s_abort) break;
          if (GATHER) fence_proxy_async_smem();  // cp.async writes -> tensor core reads
          tc::fence_after();
          const uint32_t sa0 = smem_u32(ring + (size_t)s * kStage);
          const uint32_t sb0 = sa0 + kATiles * kA;
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
#pragma unroll
            for (int step = 0; step < 4; ++step) {
              const uint64_t bd = tc::smem_desc(sb0 + j * kBt + step * 32, 16, 1024);
#pragma unroll
              for (int a = 0; a < NACC; ++a) {
                const uint64_t ad = MN ? tc::smem_desc(sa0 + a * kA + step * 4096, 1024, 2048)
                                       : tc::smem_desc(sa0 + (j * NMAT + a) * kA + step * 32, 16, 1024);
                tc::mma(tmem + a * N2, ad, bd, idesc, !(kb == kb0 && j == 0 && step == 0));
              }
            }
          }
          tc::commit(&empty[s]);
          issued = true;
        }
        if (!ok) {
          set_device_error(g.err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
        tc::commit(dfull);
        issued = true;
      }
      __syncwarp();
      // epilogue: every warp of 4..7 reads its 32 rows of each accumulator and
      // adds the lo half of the columns to the hi half
      const bool ok = __all_sync(SFFN_FULL_MASK, mbar_wait_bounded(dfull, (uint32_t)(ui & 1)));
      if (!ok || __any_sync(SFFN_FULL_MASK, *(volatile int*)&s_abort)) {
        if (!ok && lane == 0) {
          set_device_error(g.err, SFFN_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
        break;
      }
      tc::fence_after();
      const uint32_t tl = tmem + ((uint32_t)(ew * 32) << 16);
#pragma unroll
      for (int a = 0; a < NACC; ++a) {
        // slot cta + mt, token-major: token n's value of output row r at
        // n * tile_rows + r (MN-major: r = a * 128 + the lane's row), so each
        // store of a warp writes 32 consecutive rows of one token
        float* dst = MN ? g.D + (size_t)(cta + mt) * p.tile_rows * NPAD + a * kTileM + ew * 32 + lane
                        : g.D + (size_t)a * g.dmat_stride + (size_t)(cta + mt) * kTileM * NPAD + ew * 32 + lane;
#pragma unroll
        for (int c0 = 0; c0 < NPAD; c0 += 16) {
          float vh[16], vl[16];
          tc::ld16(tl + (uint32_t)(a * N2 + c0), vh);
          tc::ld16(tl + (uint32_t)(a * N2 + NPAD + c0), vl);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) dst[(size_t)(c0 + i) * p.tile_rows] = vh[i] + vl[i];
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty);
    }
    // let every issued MMA finish before tensor memory is released
    if (warp == 4 && lane == 0 && issued) {
      tc::commit(drain);
      mbar_wait_bounded(drain, 0u);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 4) tc::dealloc(tmem, kCols);
}

// ---------------------------------------------------------------- finishers

template <typename T>
__device__ __forceinline__ void split16(float v, T& hi, T& lo);

template <>
__device__ __forceinline__ void split16<__nv_bfloat16>(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

template <>
__device__ __forceinline__ void split16<__half>(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

// out[hl][n][k] for n < npad, k < K: hi/lo parts of in[n][k] (n < B), zero rows n >= B.
template <typename T>
__global__ void k_b_split(const float* in, int B, int K, int npad, T* out) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t total = (size_t)npad * K;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int n = (int)(i / K);
    const float v = n < B ? ld_dep(in + i) : 0.f;
    T hi, lo;
    split16<T>(v, hi, lo);
    out[i] = hi;
    out[total + i] = lo;
  }
}

// The partial tiles are laid out token-major, [slot][npad][tile_rows]: the
// finishers below give consecutive threads consecutive output rows of one
// token, so every load of a warp reads 128 contiguous bytes of a partial and
// every 16-bit output [npad][rows] is written coalesced too.

// Partials of output row `row` (tile mt = row / tile_rows): the CTAs b0..b1
// that touched its tile, slot b + mt each.
struct RowSlots {
  const float* q;  // the row's value of token 0 in slot b0 + mt
  size_t slot;     // floats per slot
  int nb;          // b1 - b0 + 1, 0 for an empty product
};

__device__ __forceinline__ RowSlots row_slots(const float* D, const Plan& p, int row, int npad) {
  RowSlots r;
  r.slot = (size_t)p.tile_rows * npad;
  r.nb = 0;
  r.q = D;
  if (p.total == 0) return r;
  const int mt = row / p.tile_rows, rr = row % p.tile_rows;
  const int b0 = cta_of(p, (long long)mt * p.kblocks), b1 = cta_of(p, (long long)(mt + 1) * p.kblocks - 1);
  r.nb = b1 - b0 + 1;
  r.q = D + (size_t)(b0 + mt) * r.slot + rr;
  return r;
}

// Tokens n0..n0+T-1 of the row (those below nvalid; the others stay 0): each
// token's partials added in CTA order, the loads of KB CTAs for all T tokens
// in flight together.
template <int T, int KB>
__device__ __forceinline__ void sum_partials(const RowSlots& r, int n0, int nvalid, int tile_rows, float (&acc)[T]) {
#pragma unroll
  for (int e = 0; e < T; ++e) acc[e] = 0.f;
  const float* q = r.q + (size_t)n0 * tile_rows;
  for (int b = 0; b < r.nb; b += KB) {
    float v[KB][T];
#pragma unroll
    for (int k = 0; k < KB; ++k)
#pragma unroll
      for (int e = 0; e < T; ++e)
        v[k][e] = b + k < r.nb && n0 + e < nvalid ? ld_dep(q + (size_t)(b + k) * r.slot + (size_t)e * tile_rows) : 0.f;
#pragma unroll
    for (int k = 0; k < KB; ++k)
      if (b + k < r.nb)
#pragma unroll
        for (int e = 0; e < T; ++e) acc[e] += v[k][e];
  }
}

// hid[n][j] = ReLU(sum_kq D[kq][n][j] + b1[j]) as hi/lo parts [2][npad][h].
// Thread i = n * h + j.
template <typename T>
__global__ void k_b_hidden_fin(const float* D, int d, int grid, int npad, int h, int B, const float* b1, T* out) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= npad * h) return;
  const int n = i / h, j = i % h;
  float v = 0.f;
  if (n < B) {
    const Plan p = make_plan(false, h, d, grid, ksub_contig(d));  // the hidden product's plan (K = d)
    float a[1];
    sum_partials<1, 16>(row_slots(D, p, j, npad), n, B, p.tile_rows, a);
    v = relu_nan(a[0] + (b1 ? b1[j] : 0.f));
  }
  T hi, lo;
  split16<T>(v, hi, lo);
  out[(size_t)n * h + j] = hi;
  out[(size_t)npad * h + (size_t)n * h + j] = lo;
}

// nmask[n][w] for every token n < B, and the union word unmask[w]. A block
// of 256 threads takes two mask words, four warps each; lane = row of the
// word, warp q of a word takes tokens 8q..8q+7 (one ballot per token) and the
// four warps' unions are joined in shared memory.
__global__ void __launch_bounds__(256)
    k_b_scores_fin(const float* D, int h, int grid, int npad, int nw, int B, const float* b2, float thres,
                   uint32_t* nmask, uint32_t* unmask) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint32_t s_uni[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * 2 + (warp >> 2), q = warp & 3;
  uint32_t uni = 0;
  if (w < nw && q * 8 < B) {
    const int row = w * 32 + lane;
    const Plan p = make_plan(false, nw * 32, h, grid, ksub_contig(h));  // the scores product's plan (K = h)
    const RowSlots r = row_slots(D, p, row, npad);
    float acc[8];
    sum_partials<8, 4>(r, q * 8, B, p.tile_rows, acc);
    const float bias = b2 ? b2[row] : 0.f;
    uint32_t mine = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t m = __ballot_sync(SFFN_FULL_MASK, q * 8 + e < B && acc[e] + bias >= thres);  // NaN: false
      if (lane == e) mine = m;
      uni |= m;
    }
    if (lane < 8 && q * 8 + lane < B) nmask[(size_t)(q * 8 + lane) * nw + w] = mine;
  }
  if (lane == 0) s_uni[warp] = uni;
  __syncthreads();
  if ((warp & 3) == 0 && lane == 0 && w < nw)
    unmask[w] = s_uni[warp] | s_uni[warp + 1] | s_uni[warp + 2] | s_uni[warp + 3];
}

// Writes the ascending active list to out (s_words / s_off from
// scan_mask_words): warp k takes a run of consecutive words, 32 at a time with
// one word and its list offset per lane, and walks them by shuffles; lane l
// tests bit l of the word and the set lanes store their entries side by side
// (list position = the word's offset + the set bits below the lane).
__device__ __forceinline__ void extract_list_ballot(const uint32_t* s_words, const int* s_off, int nw,
                                                    int32_t* out) {
  constexpr int kWarps = kViewThreadsB / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (nw + kWarps - 1) / kWarps;
  const int w0 = min(nw, warp * per), w1 = min(nw, w0 + per);
  const uint32_t below = (1u << lane) - 1u;
  for (int c = w0; c < w1; c += 32) {
    const int n = min(32, w1 - c);
    const uint32_t ml = lane < n ? s_words[c + lane] : 0u;
    const int pl = lane < n ? s_off[c + lane] : 0;
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const uint32_t m = __shfl_sync(SFFN_FULL_MASK, ml, k);
      const int p = __shfl_sync(SFFN_FULL_MASK, pl, k);
      if ((m >> lane) & 1u) out[p + __popc(m & below)] = (c + k) * 32 + lane;
    }
  }
}

// Views: block b < B expands token b's mask (index list, count, group mask);
// block B expands the union mask, forming it first (OR over tokens) unless
// the scores finisher already wrote it (union_ready).
__global__ void __launch_bounds__(kViewThreadsB)
    k_b_views(const uint32_t* nmask, int B, int nw, int f, int n_groups, int G, int gwords, int32_t* idx,
              int32_t* count, uint32_t* gmask, uint32_t* unmask, int32_t* uidx, int32_t* ucount, uint32_t* ugmask,
              bool union_ready) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* s_words = reinterpret_cast<uint32_t*>(smem);
  int* s_off = reinterpret_cast<int*>(s_words + nw);
  __shared__ int s_tmp[kViewThreadsB / 32];
  const int b = blockIdx.x;
  const uint32_t* src;
  if (b < B) {
    src = nmask + (size_t)b * nw;
  } else if (union_ready) {
    src = unmask;
  } else {
    // union words into the union mask output, then scanned like any token
    for (int w = threadIdx.x; w < nw; w += kViewThreadsB) {
      uint32_t m = 0;
      for (int n = 0; n < B; ++n) m |= ld_dep(nmask + (size_t)n * nw + w);
      unmask[w] = m;
    }
    __syncthreads();
    __threadfence_block();
    src = unmask;
  }
  const int total = scan_mask_words<kViewThreadsB>(src, nw, s_words, s_off, s_tmp);
  if (b < B) {
    if (idx) extract_list_ballot(s_words, s_off, nw, idx + (size_t)b * f);
    if (count && threadIdx.x == 0) count[b] = total;
    if (gmask) write_group_mask<kViewThreadsB>(s_words, n_groups, G, gwords, gmask + (size_t)b * gwords);
  } else {
    extract_list_ballot(s_words, s_off, nw, uidx);
    if (threadIdx.x == 0) *ucount = total;
    if (ugmask) write_group_mask<kViewThreadsB>(s_words, n_groups, G, gwords, ugmask);
  }
}

// H parts [2][npad][ldh]: h = act(g, u) for union neuron u and token n if the
// neuron is in token n's own mask, else 0; zero beyond the union and for n >= B.
// Thread i = q * ldh + u takes tokens 8q..8q+7 of union neuron u.
template <typename T, int ACT>
__global__ void k_b_act_fin(const float* Du, const float* Dg, int d, const int32_t* ucount,
                            const int32_t* uidx, const uint32_t* nmask, int nw, int npad, int B, int ldh,
                            int grid, T* H) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (npad / 8) * ldh) return;
  const int n0 = (i / ldh) * 8, u = i % ldh;
  const int U = ld_dep(ucount);
  if (u >= (U + kTileK - 1) / kTileK * kTileK) return;  // the down product reads no further
  float v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = 0.f;
  if (u < U && n0 < B) {
    const Plan p = make_plan(false, U, d, grid, ksub_gather(d, act_gated(ACT) ? 2 : 1));  // the up/gate plan
    float su[8], sg[8];
    sum_partials<8, 4>(row_slots(Du, p, u, npad), n0, B, p.tile_rows, su);
    if (act_gated(ACT)) {
      sum_partials<8, 4>(row_slots(Dg, p, u, npad), n0, B, p.tile_rows, sg);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) sg[e] = 0.f;
    }
    const int slot = ld_dep(uidx + u);
    uint32_t mw[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mw[e] = n0 + e < B ? ld_dep(nmask + (size_t)(n0 + e) * nw + (slot >> 5)) : 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if ((mw[e] >> (slot & 31)) & 1u) v[e] = neuron_act<ACT>(su[e], sg[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const size_t o = (size_t)(n0 + e) * ldh + u;
    T hi, lo;
    split16<T>(v[e], hi, lo);
    H[o] = hi;
    H[(size_t)npad * ldh + o] = lo;
  }
}

// y[n][c] = sum_kq D[kq][n][c]; x_out = x + y. Thread i = q * d + c takes
// tokens 2q and 2q + 1 of output row c.
__global__ void k_b_y_fin(const float* D, const int32_t* ucount, int d, int npad, int B, int grid, const float* x,
                          float* y, float* x_out) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (B + 1) / 2 * d) return;
  const int n0 = (i / d) * 2, c = i % d;
  float xv[2] = {0.f, 0.f};
  if (x_out) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (n0 + e < B) xv[e] = ld_dep(x + (size_t)(n0 + e) * d + c);
  }
  const int U = ld_dep(ucount);
  const Plan p = make_plan(true, U, d, grid, 1, msub_down(d));
  float s[2];
  sum_partials<2, 8>(row_slots(D, p, c, npad), n0, B, p.tile_rows, s);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    if (n0 + e < B) {
      const size_t o = (size_t)(n0 + e) * d + c;
      y[o] = s[e];
      if (x_out) x_out[o] = xv[e] + s[e];
    }
  }
}

}  // namespace

// ---------------------------------------------------------------- host side

namespace {

int npad_of(int B) { return B <= 16 ? 16 : 32; }
int gemm_grid(const sffn_layer& L) { return L.num_sms; }

size_t rows_bound(const sffn_layer& L, int m_tiles_max) {
  return ((size_t)gemm_grid(L) + (size_t)m_tiles_max) * kTileM;  // partial slots < CTAs + tiles
}

template <bool MN, int NMAT, int NPAD, int KSUB, int MSUB>
size_t gemm_stage_bytes() {
  const size_t a_tiles = MN ? MSUB : (size_t)KSUB * NMAT;
  return a_tiles * kTileM * kTileK * 2 + (size_t)KSUB * 2 * NPAD * kTileK * 2;
}

template <bool MN, int NMAT, int NPAD, int KSUB, int MSUB>
int gemm_stages() {
  return (int)std::min<size_t>(8, (kGemmSmemBudget - 2048) / gemm_stage_bytes<MN, NMAT, NPAD, KSUB, MSUB>());
}

template <bool MN, int NMAT, int NPAD, int KSUB, int MSUB>
size_t gemm_smem() {
  const int stages = gemm_stages<MN, NMAT, NPAD, KSUB, MSUB>();
  return 1024 + (size_t)stages * gemm_stage_bytes<MN, NMAT, NPAD, KSUB, MSUB>() + (size_t)(3 * stages + 3) * 8;
}

template <bool MN, int NMAT, int NPAD, int KSUB, int MSUB>
constexpr bool gemm_stage_bytes_ok() {
  return 2 * ((MN ? MSUB : KSUB * NMAT) * kTileM * kTileK * 2 + KSUB * 2 * NPAD * kTileK * 2) <= kGemmSmemBudget - 2048;
}

template <bool MN, int NMAT, int NPAD, bool GATHER, int KSUB, int MSUB>
cudaError_t set_gemm_attr_one() {
  static_assert(gemm_stage_bytes_ok<MN, NMAT, NPAD, KSUB, MSUB>(), "two ring stages must fit");
  auto* k = k_tc_gemm<MN, NMAT, NPAD, GATHER, KSUB, MSUB>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gemm_smem<MN, NMAT, NPAD, KSUB, MSUB>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

template <bool MN, int NMAT, bool GATHER, int KSUB, int MSUB>
cudaError_t set_gemm_attr() {
  cudaError_t e = set_gemm_attr_one<MN, NMAT, 16, GATHER, KSUB, MSUB>();
  return e != cudaSuccess ? e : set_gemm_attr_one<MN, NMAT, 32, GATHER, KSUB, MSUB>();
}

template <bool MN, int NMAT, bool GATHER, int KSUB, int MSUB>
cudaError_t launch_gemm(const sffn_layer& L, int npad, const GemmArgs& g, cudaStream_t st) {
  const bool bf = L.desc.wdtype == SFFN_BF16;
  if (npad == 16)
    return launch_ex(k_tc_gemm<MN, NMAT, 16, GATHER, KSUB, MSUB>, dim3(g.grid), dim3(kGemmThreads),
                     gemm_smem<MN, NMAT, 16, KSUB, MSUB>(), st, true, 1, g, bf,
                     gemm_stages<MN, NMAT, 16, KSUB, MSUB>());
  return launch_ex(k_tc_gemm<MN, NMAT, 32, GATHER, KSUB, MSUB>, dim3(g.grid), dim3(kGemmThreads),
                   gemm_smem<MN, NMAT, 32, KSUB, MSUB>(), st, true, 1, g, bf, gemm_stages<MN, NMAT, 32, KSUB, MSUB>());
}

// Contiguous rows (hidden, scores): K steps of ksub_contig(K) blocks.
cudaError_t launch_contig(const sffn_layer& L, int npad, const GemmArgs& g, cudaStream_t st) {
  return ksub_contig(g.other) == 4 ? launch_gemm<false, 1, false, 4, 1>(L, npad, g, st)
                                   : launch_gemm<false, 1, false, 1, 1>(L, npad, g, st);
}

// Gathered union rows of up (and gate): K steps of ksub_gather(d, nmat) blocks.
cudaError_t launch_upgate(const sffn_layer& L, int npad, bool gated, const GemmArgs& g, cudaStream_t st) {
  const int ks = ksub_gather(g.other, gated ? 2 : 1);
  if (gated) return ks == 2 ? launch_gemm<false, 2, true, 2, 1>(L, npad, g, st)
                            : launch_gemm<false, 2, true, 1, 1>(L, npad, g, st);
  return ks == 2 ? launch_gemm<false, 1, true, 2, 1>(L, npad, g, st) : launch_gemm<false, 1, true, 1, 1>(L, npad, g, st);
}

// Gathered union rows of downT (MN-major): output tiles of msub_down(d) x 128 rows.
cudaError_t launch_down(const sffn_layer& L, int npad, const GemmArgs& g, cudaStream_t st) {
  const int ms = msub_down(g.other);
  return ms == 4 ? launch_gemm<true, 1, true, 1, 4>(L, npad, g, st)
                 : (ms == 2 ? launch_gemm<true, 1, true, 1, 2>(L, npad, g, st)
                            : launch_gemm<true, 1, true, 1, 1>(L, npad, g, st));
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a row-major 16-bit matrix [rows][inner] (row pitch
// inner * 2 bytes, a multiple of 16) read in boxes of 64 x box_rows elements
// with the 128-byte swizzle. Rows past the end read as zero.
cudaError_t encode_rows(CUtensorMap* m, const void* base, bool bf16, uint64_t inner, uint64_t rows,
                        uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

BatchWs batch_ws_layout(const sffn_layer& L, int B) {
  BatchWs w;
  const int npad = 32;  // sized for the largest padding
  const size_t d = L.desc.d, f = L.desc.f, h = L.desc.h;
  const size_t fpad = (f + kTileK - 1) / kTileK * kTileK;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = (off + bytes + 255) & ~(size_t)255;
    return o;
  };
  (void)B;
  w.xhl = take(2 * npad * d * 2);
  w.dh = take(rows_bound(L, (int)((h + kTileM - 1) / kTileM)) * npad * 4);
  w.hidhl = take(2 * npad * h * 2);
  w.ds = take(rows_bound(L, (int)((f + kTileM - 1) / kTileM)) * npad * 4);
  w.unmask = take((f / 32) * 4);
  w.uidx = take(f * 4);
  w.ucount = take(256);
  w.dug = take(2 * rows_bound(L, (int)((f + kTileM - 1) / kTileM)) * npad * 4);
  w.hhl = take(2 * npad * fpad * 2);
  // down partials: slots < CTAs + tiles, tile_rows = msub_down(d) * 128
  w.dy = take(((size_t)gemm_grid(L) * kTileM * msub_down((int)d) + d) * npad * 4);
  w.total = off;
  return w;
}

bool batch_supported(const sffn_layer& L, std::string* why) {
  if (L.desc.ffn_format != SFFN_FFN_ROWS) {
    if (why) *why = "batched calls need 16-bit FFN rows (8-bit and 4-bit rows run at B = 1)";
    return false;
  }
  if (L.desc.wdtype == SFFN_F32) {
    if (why) *why = "batched calls need 16-bit weights (fp16 or bf16)";
    return false;
  }
  if (L.desc.d % kTileM || L.desc.h % kTileK) {
    if (why) *why = "batched calls need d a multiple of 128 and h a multiple of 64";
    return false;
  }
  return true;
}

cudaError_t configure_batch_kernels(const sffn_layer& L) {
  if (!batch_supported(L, nullptr)) return cudaSuccess;
  cudaError_t e;
  if (!tensor_map_encoder()) return cudaErrorNotSupported;
  if ((e = set_gemm_attr<false, 1, false, 1, 1>())) return e;
  if ((e = set_gemm_attr<false, 1, false, 4, 1>())) return e;
  if ((e = set_gemm_attr<false, 1, true, 1, 1>())) return e;
  if ((e = set_gemm_attr<false, 1, true, 2, 1>())) return e;
  if ((e = set_gemm_attr<false, 2, true, 1, 1>())) return e;
  if ((e = set_gemm_attr<false, 2, true, 2, 1>())) return e;
  if ((e = set_gemm_attr<true, 1, true, 1, 1>())) return e;
  if ((e = set_gemm_attr<true, 1, true, 1, 2>())) return e;
  return set_gemm_attr<true, 1, true, 1, 4>();
}

// Records the layer's trace event for slot k (if any) around `launch`.
template <typename F>
cudaError_t traced_b(const sffn_layer& L, int k, cudaStream_t st, F&& launch) {
  cudaError_t e = cudaSuccess;
  if (L.trace_begin[k]) e = cudaEventRecord(L.trace_begin[k], st);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess && L.trace_end[k]) e = cudaEventRecord(L.trace_end[k], st);
  return e;
}

cudaError_t launch_batch_views(const sffn_layer& L, const sffn_masks* m, int B, uint32_t* unmask, int32_t* uidx,
                               int32_t* ucount, bool predict, bool union_ready, cudaStream_t st) {
  const int nw = L.nwords;
  return launch_ex(k_b_views, dim3(B + 1), dim3(kViewThreadsB), (size_t)nw * 8, st, true, 1,
                   static_cast<const uint32_t*>(m->nmask), B, nw, L.desc.f, L.n_groups, L.desc.group_size, L.gwords,
                   predict ? m->idx : nullptr, predict ? m->count : nullptr, predict ? m->gmask : nullptr, unmask, uidx,
                   ucount, m->ugmask, union_ready);
}

cudaError_t launch_batch(const sffn_layer& L, const float* x, int B, float thres, const sffn_masks* m, bool predict,
                         bool forward, float* y, float* x_out, void* ws, cudaStream_t st) {
  const BatchWs w = batch_ws_layout(L, B);
  char* base = static_cast<char*>(ws);
  const int npad = npad_of(B);
  const int d = L.desc.d, f = L.desc.f, h = L.desc.h, nw = L.nwords;
  const int fpad = (f + kTileK - 1) / kTileK * kTileK;
  const bool bf = L.desc.wdtype == SFFN_BF16;
  const int grid = gemm_grid(L);
  uint32_t* unmask = m->unmask ? m->unmask : reinterpret_cast<uint32_t*>(base + w.unmask);
  int32_t* uidx = m->uidx ? m->uidx : reinterpret_cast<int32_t*>(base + w.uidx);
  int32_t* ucount = m->ucount ? m->ucount : reinterpret_cast<int32_t*>(base + w.ucount);
  cudaError_t e = cudaSuccess;
  // x -> hi/lo parts [2][npad][d]
  void* xhl = base + w.xhl;
  const int split_blocks = std::min(1024, (npad * d + 255) / 256);
  if (bf)
    e = launch_ex(k_b_split<__nv_bfloat16>, dim3(split_blocks), dim3(256), 0, st, true, 1, x, B, d, npad,
                  static_cast<__nv_bfloat16*>(xhl));
  else
    e = launch_ex(k_b_split<__half>, dim3(split_blocks), dim3(256), 0, st, true, 1, x, B, d, npad,
                  static_cast<__half*>(xhl));
  if (e != cudaSuccess) return e;

  if (predict) {
    // hidden: D[h x N] = W1 . X^T over K = d
    GemmArgs g{};
    g.A0 = static_cast<const unsigned char*>(L.W1);
    g.fixed_count = h;
    g.other = d;
    g.lda = d;
    g.Bhl = static_cast<const unsigned char*>(xhl);
    g.ldb = d;
    g.D = reinterpret_cast<float*>(base + w.dh);
    g.grid = grid;
    g.err = L.err;
    e = encode_rows(&g.tmA, L.W1, bf, d, h, kTileM);
    if (e == cudaSuccess) e = encode_rows(&g.tmB, xhl, bf, d, 2 * npad, 2 * npad);
    if (e == cudaSuccess) e = traced_b(L, 0, st, [&] { return launch_contig(L, npad, g, st); });
    if (e != cudaSuccess) return e;
    void* hidhl = base + w.hidhl;
    const int hb = (npad * h + 255) / 256;
    const float* b1 = L.has_b1 ? L.b1 : nullptr;
    if (bf)
      e = launch_ex(k_b_hidden_fin<__nv_bfloat16>, dim3(hb), dim3(256), 0, st, true, 1,
                    static_cast<const float*>(g.D), d, grid, npad, h, B, b1,
                    static_cast<__nv_bfloat16*>(hidhl));
    else
      e = launch_ex(k_b_hidden_fin<__half>, dim3(hb), dim3(256), 0, st, true, 1, static_cast<const float*>(g.D),
                    d, grid, npad, h, B, b1, static_cast<__half*>(hidhl));
    if (e != cudaSuccess) return e;
    // scores: D[f x N] = W2 . HID^T over K = h
    GemmArgs s{};
    s.A0 = static_cast<const unsigned char*>(L.W2);
    s.fixed_count = f;
    s.other = h;
    s.lda = h;
    s.Bhl = static_cast<const unsigned char*>(hidhl);
    s.ldb = h;
    s.D = reinterpret_cast<float*>(base + w.ds);
    s.grid = grid;
    s.err = L.err;
    e = encode_rows(&s.tmA, L.W2, bf, h, f, kTileM);
    if (e == cudaSuccess) e = encode_rows(&s.tmB, hidhl, bf, h, 2 * npad, 2 * npad);
    if (e == cudaSuccess) e = traced_b(L, 1, st, [&] { return launch_contig(L, npad, s, st); });
    if (e != cudaSuccess) return e;
    const float* b2 = L.has_b2 ? L.b2 : nullptr;
    e = launch_ex(k_b_scores_fin, dim3((nw + 1) / 2), dim3(256), 0, st, true, 1, static_cast<const float*>(s.D), h,
                  grid, npad, nw, B, b2, thres, m->nmask, unmask);
    if (e != cudaSuccess) return e;
  }
  // per-token views (when predicting) and the union mask with its views
  e = launch_ex(k_b_views, dim3(B + 1), dim3(kViewThreadsB), (size_t)nw * 8, st, true, 1,
                static_cast<const uint32_t*>(m->nmask), B, nw, f, L.n_groups, L.desc.group_size, L.gwords,
                predict ? m->idx : nullptr, predict ? m->count : nullptr, predict ? m->gmask : nullptr, unmask, uidx,
                ucount, m->ugmask, predict);
  if (e != cudaSuccess || !forward) return e;

  // up/gate over the union rows: D[U x N] = {up, gate} . X^T over K = d
  const bool gated = act_gated(L.desc.act);
  const size_t dmat = rows_bound(L, (f + kTileM - 1) / kTileM) * npad;
  GemmArgs u{};
  u.A0 = static_cast<const unsigned char*>(L.up);
  u.A1 = gated ? static_cast<const unsigned char*>(L.gate) : nullptr;
  u.rows = uidx;
  u.count_dev = ucount;
  u.other = d;
  u.lda = d;
  u.Bhl = static_cast<const unsigned char*>(xhl);
  u.ldb = d;
  u.D = reinterpret_cast<float*>(base + w.dug);
  u.dmat_stride = dmat;
  u.grid = grid;
  u.err = L.err;
  e = encode_rows(&u.tmB, xhl, bf, d, 2 * npad, 2 * npad);
  if (e == cudaSuccess) e = traced_b(L, 2, st, [&] { return launch_upgate(L, npad, gated, u, st); });
  if (e != cudaSuccess) return e;
  // activation with each token's own mask -> H parts [2][npad][fpad]
  void* hhl = base + w.hhl;
  const int ab = ((npad / 8) * fpad + 255) / 256;
#define SFFN_ACT_LAUNCH(T, A)                                                                                     \
  launch_ex(k_b_act_fin<T, A>, dim3(ab), dim3(256), 0, st, true, 1, static_cast<const float*>(u.D),              \
            static_cast<const float*>(u.D + dmat), d, static_cast<const int32_t*>(ucount),                        \
            static_cast<const int32_t*>(uidx), static_cast<const uint32_t*>(m->nmask), nw, npad, B, fpad, grid, \
            static_cast<T*>(hhl))
  switch (L.desc.act) {
    case SFFN_ACT_RELU: e = bf ? SFFN_ACT_LAUNCH(__nv_bfloat16, SFFN_ACT_RELU) : SFFN_ACT_LAUNCH(__half, SFFN_ACT_RELU); break;
    case SFFN_ACT_REGLU: e = bf ? SFFN_ACT_LAUNCH(__nv_bfloat16, SFFN_ACT_REGLU) : SFFN_ACT_LAUNCH(__half, SFFN_ACT_REGLU); break;
    case SFFN_ACT_RELU2: e = bf ? SFFN_ACT_LAUNCH(__nv_bfloat16, SFFN_ACT_RELU2) : SFFN_ACT_LAUNCH(__half, SFFN_ACT_RELU2); break;
    default: e = bf ? SFFN_ACT_LAUNCH(__nv_bfloat16, SFFN_ACT_SWIGLU) : SFFN_ACT_LAUNCH(__half, SFFN_ACT_SWIGLU); break;
  }
#undef SFFN_ACT_LAUNCH
  if (e != cudaSuccess) return e;
  // down: D[d x N] = downT^T (MN-major, K = union rows) . H^T
  GemmArgs dn{};
  dn.A0 = static_cast<const unsigned char*>(L.downT);
  dn.rows = uidx;
  dn.count_dev = ucount;
  dn.other = d;
  dn.lda = d;
  dn.Bhl = static_cast<const unsigned char*>(hhl);
  dn.ldb = fpad;
  dn.D = reinterpret_cast<float*>(base + w.dy);
  dn.grid = grid;
  dn.err = L.err;
  e = encode_rows(&dn.tmB, hhl, bf, fpad, 2 * npad, 2 * npad);
  if (e == cudaSuccess) e = traced_b(L, 3, st, [&] { return launch_down(L, npad, dn, st); });
  if (e != cudaSuccess) return e;
  return launch_ex(k_b_y_fin, dim3(((B + 1) / 2 * d + 255) / 256), dim3(256), 0, st, true, 1, static_cast<const float*>(dn.D),
                   static_cast<const int32_t*>(ucount), d, npad, B, grid, x, y, x_out);
}

}  // namespace sffn
