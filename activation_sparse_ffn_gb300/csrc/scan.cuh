// Block-wide scans over a neuron bitmask: word offsets of the ascending
// active-slot list, the slice of that list a thread block owns, and the
// group bitmask (a group is active iff any of its slots is).
#pragma once

#include "common.cuh"

namespace sffn {

// Exclusive prefix sum of one int per thread over a block of NT threads.
// s_tmp holds NT/32 ints. Returns the exclusive prefix; *total gets the sum.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_tmp, int* total) {
  static_assert(NT % 32 == 0 && NT <= 1024, "block size");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(SFFN_FULL_MASK, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < NT / 32) ? s_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(SFFN_FULL_MASK, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) s_tmp[lane] = w;
  }
  __syncthreads();
  const int before = warp ? s_tmp[warp - 1] : 0;
  *total = s_tmp[NT / 32 - 1];
  __syncthreads();
  return before + x - v;
}

// Most mask words a layer has: f <= 1024 groups of at most 64 slots.
constexpr int kMaxMaskWords = 2048;

// Loads nw mask words into s_words and writes each word's offset in the
// ascending active list into s_off. Returns the number of active slots.
// Every thread first requests all of its words at once (coalesced,
// independent loads: one L2 round trip instead of one per word), then counts
// a contiguous range of them from shared memory.
template <int NT>
__device__ __forceinline__ int scan_mask_words(const uint32_t* nmask, int nw, uint32_t* s_words,
                                               int* s_off, int* s_tmp) {
  constexpr int kIter = (kMaxMaskWords + NT - 1) / NT;
  uint32_t v[kIter];
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int w = (int)threadIdx.x + i * NT;
    v[i] = w < nw ? ld_dep(nmask + w) : 0u;  // written by the previous kernel
  }
#pragma unroll
  for (int i = 0; i < kIter; ++i) {
    const int w = (int)threadIdx.x + i * NT;
    if (w < nw) s_words[w] = v[i];
  }
  __syncthreads();
  const int per = (nw + NT - 1) / NT;
  const int w0 = min(nw, (int)threadIdx.x * per), w1 = min(nw, w0 + per);
  int local = 0;
  for (int w = w0; w < w1; ++w) local += __popc(s_words[w]);
  int total;
  int off = block_exclusive_scan<NT>(local, s_tmp, &total);
  for (int w = w0; w < w1; ++w) {
    s_off[w] = off;
    off += __popc(s_words[w]);
  }
  __syncthreads();
  return total;
}

// Writes the active slots with list positions in [lo, hi) to out[p - lo]
// (ascending order). Needs s_words / s_off from scan_mask_words.
template <int NT>
__device__ __forceinline__ void extract_slice(const uint32_t* s_words, const int* s_off, int nw, int lo, int hi,
                                              int32_t* out) {
  for (int w = threadIdx.x; w < nw; w += NT) {
    uint32_t m = s_words[w];
    int p = s_off[w];
    if (p >= hi || p + __popc(m) <= lo) continue;
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1;
      if (p >= lo && p < hi) out[p - lo] = w * 32 + b;
      ++p;
    }
  }
}

// Group bitmask from the neuron words: group g covers words
// [g*G/32, (g+1)*G/32). Writes gwords words.
template <int NT>
__device__ __forceinline__ void write_group_mask(const uint32_t* s_words, int n_groups, int G, int gwords,
                                                 uint32_t* __restrict__ gmask) {
  const int wpg = G / 32;
  for (int g = threadIdx.x; g < gwords * 32; g += NT) {
    bool a = false;
    if (g < n_groups) {
      for (int k = 0; k < wpg; ++k) a |= (s_words[g * wpg + k] != 0u);
    }
    const uint32_t word = __ballot_sync(SFFN_FULL_MASK, a);
    if ((threadIdx.x & 31) == 0) gmask[g >> 5] = word;
  }
}

}  // namespace sffn
