// Setup-time packing into the grouped, neuron-major layout: slot s of every
// per-neuron array holds original neuron perm[s] (the neuron table of
// PowerInfer §5.2), so the co-activation groups of KAIROX (核心方法 items 1 and
// 3) are contiguous slot ranges; down is transposed so that a neuron's output
// column becomes one contiguous row. Not on the hot path.
#include "common.cuh"
#include "internal.h"

namespace sffn {

namespace {

// Marks perm values in a bitmap; an out-of-range or repeated value flags
// SFFN_ERR_DEVICE.
__global__ void k_perm_check(const int32_t* __restrict__ perm, int f, uint32_t* __restrict__ bitmap,
                             uint32_t* __restrict__ err) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= f) return;
  const int n = perm[s];
  if (n < 0 || n >= f) {
    set_device_error(err, SFFN_ERR_DEVICE);
    return;
  }
  const uint32_t bit = 1u << (n & 31);
  if (atomicOr(&bitmap[n >> 5], bit) & bit) set_device_error(err, SFFN_ERR_DEVICE);
}

// dst row s = src row perm[s] (identity when perm is null); rows of
// row_bytes (a multiple of 16) copied as 16-byte vectors.
__global__ void k_gather_rows(unsigned char* __restrict__ dst, const unsigned char* __restrict__ src,
                              const int32_t* __restrict__ perm, int rows, size_t row_bytes,
                              uint32_t* __restrict__ err) {
  const int s = blockIdx.x;
  const int n = perm ? perm[s] : s;
  if (n < 0 || n >= rows) {
    if (threadIdx.x == 0) set_device_error(err, SFFN_ERR_DEVICE);
    return;
  }
  const uint4* sp = reinterpret_cast<const uint4*>(src + (size_t)n * row_bytes);
  uint4* dp = reinterpret_cast<uint4*>(dst + (size_t)s * row_bytes);
  for (size_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x) dp[i] = sp[i];
}

// dst row s = the 4-bit packing of int8 code row perm[s] of src [rows][d]
// (identity when perm is null): byte i = (code 2i & 15) | (code 2i+1 & 15) << 4.
// A code outside [-8, 7] or an out-of-range perm value flags SFFN_ERR_DEVICE.
__global__ void k_pack_q4_rows(uint8_t* __restrict__ dst, const int8_t* __restrict__ src,
                               const int32_t* __restrict__ perm, int rows, int d, uint32_t* __restrict__ err) {
  const int s = blockIdx.x;
  const int n = perm ? perm[s] : s;
  if (n < 0 || n >= rows) {
    if (threadIdx.x == 0) set_device_error(err, SFFN_ERR_DEVICE);
    return;
  }
  const int8_t* sp = src + (size_t)n * d;
  uint8_t* dp = dst + (size_t)s * (d / 2);
  for (int i = threadIdx.x; i < d / 2; i += blockDim.x) {
    const int c0 = sp[2 * i], c1 = sp[2 * i + 1];
    if (c0 < -8 || c0 > 7 || c1 < -8 || c1 > 7) set_device_error(err, SFFN_ERR_DEVICE);
    dp[i] = (uint8_t)((c0 & 15) | ((c1 & 15) << 4));
  }
}

__global__ void k_gather_f32(float* __restrict__ dst, const float* __restrict__ src, const int32_t* __restrict__ perm,
                             int n) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < n) {
    const int k = perm ? perm[s] : s;
    dst[s] = (k >= 0 && k < n) ? src[k] : 0.f;
  }
}

__global__ void k_iota(int32_t* __restrict__ out, int n) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < n) out[s] = s;
}

// src [R][C] -> dst [C][R] through 32x32 shared-memory tiles.
template <typename T>
__global__ void k_transpose(T* __restrict__ dst, const T* __restrict__ src, int R, int C) {
  __shared__ T tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = src[(size_t)r * C + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < C && r < R) dst[(size_t)c * R + r] = tile[threadIdx.x][i];
  }
}

// Transpose of the FFN's down matrix as given to the pack call, moved as raw
// elements: 4 or 2 bytes for plain rows, 1 byte for 8-bit and 4-bit codes
// (which arrive one int8 per code).
cudaError_t transpose(const sffn_layer& L, void* dst, const void* src, int R, int C, cudaStream_t st) {
  const dim3 grid((C + 31) / 32, (R + 31) / 32), block(32, 8);
  switch (L.fbits >= 8 ? L.fbits / 8 : 1) {
    case 4:
      k_transpose<float><<<grid, block, 0, st>>>(static_cast<float*>(dst), static_cast<const float*>(src), R, C);
      break;
    case 2:
      k_transpose<uint16_t><<<grid, block, 0, st>>>(static_cast<uint16_t*>(dst), static_cast<const uint16_t*>(src),
                                                     R, C);
      break;
    default:
      k_transpose<uint8_t><<<grid, block, 0, st>>>(static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), R,
                                                    C);
      break;
  }
  return cudaGetLastError();
}

cudaError_t gather_rows(void* dst, const void* src, const int32_t* perm, int rows, size_t row_bytes, uint32_t* err,
                        cudaStream_t st) {
  k_gather_rows<<<rows, 256, 0, st>>>(static_cast<unsigned char*>(dst), static_cast<const unsigned char*>(src), perm,
                                      rows, row_bytes, err);
  return cudaGetLastError();
}

}  // namespace

sffn_status pack_layer(sffn_layer& L, const void* W1, const float* b1, const void* W2, const float* b2,
                       const void* up, const void* gate, const void* down, const int32_t* perm, cudaStream_t st,
                       const float* up_s, const float* gate_s, const float* down_s) {
  const int d = L.desc.d, f = L.desc.f, h = L.desc.h;
  const size_t wb = (size_t)L.wbytes, frow = ffn_row_bytes(L);
  const bool q4 = L.fbits == 4;
  const size_t in_elem = q4 ? 1 : (size_t)L.fbits / 8;  // bytes per element of the caller's up/gate/down
  cudaError_t e;
  uint32_t herr = 0;
  void* tmp = nullptr;
  uint32_t* bitmap = nullptr;
  sffn_status rc = SFFN_OK;

#define SFFN_TRY(call, what)             \
  do {                                   \
    if ((e = (call)) != cudaSuccess) {   \
      rc = cuda_fail(e, what);           \
      goto done;                         \
    }                                    \
  } while (0)

  SFFN_TRY(cudaMemsetAsync(L.err, 0, sizeof(uint32_t), st), "pack: clear error word");
  if (perm) {
    SFFN_TRY(cudaMalloc(&bitmap, (size_t)((f + 31) / 32) * 4), "pack: perm bitmap");
    SFFN_TRY(cudaMemsetAsync(bitmap, 0, (size_t)((f + 31) / 32) * 4, st), "pack: perm bitmap");
    k_perm_check<<<(f + 255) / 256, 256, 0, st>>>(perm, f, bitmap, L.err);
    SFFN_TRY(cudaGetLastError(), "pack: perm check");
    SFFN_TRY(cudaMemcpyAsync(&herr, L.err, 4, cudaMemcpyDeviceToHost, st), "pack: read error word");
    SFFN_TRY(cudaStreamSynchronize(st), "pack: perm check");
    if (herr) {
      set_error("sffn_layer_pack: perm is not a permutation of 0..f-1");
      rc = SFFN_ERR_DEVICE;
      cudaMemsetAsync(L.err, 0, sizeof(uint32_t), st);  // reported here, so cleared
      goto done;
    }
    SFFN_TRY(cudaMemcpyAsync(L.perm, perm, (size_t)f * 4, cudaMemcpyDeviceToDevice, st), "pack: perm");
  } else {
    k_iota<<<(f + 255) / 256, 256, 0, st>>>(L.perm, f);
    SFFN_TRY(cudaGetLastError(), "pack: iota");
  }

  SFFN_TRY(cudaMemcpyAsync(L.W1, W1, (size_t)h * d * wb, cudaMemcpyDeviceToDevice, st), "pack: W1");
  if (b1) {
    SFFN_TRY(cudaMemcpyAsync(L.b1, b1, (size_t)h * 4, cudaMemcpyDeviceToDevice, st), "pack: b1");
  } else {
    SFFN_TRY(cudaMemsetAsync(L.b1, 0, (size_t)h * 4, st), "pack: b1");
  }
  L.has_b1 = b1 != nullptr;
  SFFN_TRY(gather_rows(L.W2, W2, perm, f, (size_t)h * wb, L.err, st), "pack: W2");
  if (b2) {
    k_gather_f32<<<(f + 255) / 256, 256, 0, st>>>(L.b2, b2, perm, f);
    SFFN_TRY(cudaGetLastError(), "pack: b2");
  } else {
    SFFN_TRY(cudaMemsetAsync(L.b2, 0, (size_t)f * 4, st), "pack: b2");
  }
  L.has_b2 = b2 != nullptr;
  SFFN_TRY(cudaMalloc(&tmp, (size_t)f * d * in_elem), "pack: transpose buffer");
  SFFN_TRY(transpose(L, tmp, down, d, f, st), "pack: transpose down");
  if (q4) {  // codes arrive one per int8 and are stored two per byte
    k_pack_q4_rows<<<f, 256, 0, st>>>(static_cast<uint8_t*>(L.up), static_cast<const int8_t*>(up), perm, f, d, L.err);
    if (L.gate)
      k_pack_q4_rows<<<f, 256, 0, st>>>(static_cast<uint8_t*>(L.gate), static_cast<const int8_t*>(gate), perm, f, d,
                                        L.err);
    k_pack_q4_rows<<<f, 256, 0, st>>>(static_cast<uint8_t*>(L.downT), static_cast<const int8_t*>(tmp), perm, f, d,
                                      L.err);
    SFFN_TRY(cudaGetLastError(), "pack: 4-bit rows");
  } else {
    SFFN_TRY(gather_rows(L.up, up, perm, f, frow, L.err, st), "pack: up");
    if (L.gate) SFFN_TRY(gather_rows(L.gate, gate, perm, f, frow, L.err, st), "pack: gate");
    SFFN_TRY(gather_rows(L.downT, tmp, perm, f, frow, L.err, st), "pack: downT");
  }
  if (L.up_s) {  // quantized rows: each scale follows its neuron into slot order
    k_gather_f32<<<(f + 255) / 256, 256, 0, st>>>(L.up_s, up_s, perm, f);
    if (L.gate_s) k_gather_f32<<<(f + 255) / 256, 256, 0, st>>>(L.gate_s, gate_s, perm, f);
    k_gather_f32<<<(f + 255) / 256, 256, 0, st>>>(L.down_s, down_s, perm, f);
    SFFN_TRY(cudaGetLastError(), "pack: scales");
  }
  SFFN_TRY(cudaMemcpyAsync(&herr, L.err, 4, cudaMemcpyDeviceToHost, st), "pack: read error word");
  SFFN_TRY(cudaStreamSynchronize(st), "pack: synchronize");
  if (herr) {
    set_error("sffn_layer_pack: a device check failed while packing");
    rc = (sffn_status)herr;
    cudaMemsetAsync(L.err, 0, sizeof(uint32_t), st);  // reported here, so cleared
  }
#undef SFFN_TRY
done:
  if (tmp || bitmap) cudaStreamSynchronize(st);
  if (tmp) cudaFree(tmp);
  if (bitmap) cudaFree(bitmap);
  return rc;
}

}  // namespace sffn
