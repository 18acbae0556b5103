// sffn_decode_step_static_ws: the decode step without a caller workspace.
//
// Some callers cannot allocate device memory: a decode loop that must never
// stall (a device allocation can synchronize the whole GPU), a runtime that
// reaches this library only through its C ABI and has no CUDA allocator of its
// own, or a process whose memory pool forbids new allocations once serving has
// started. For them this entry point takes its scratch space from one
// file-scope device array, so it calls no allocator at all. The caller still
// owns x, y, x_out and the mask buffers.
//
// The array holds 16 MiB: the workspace of any valid layer at batch size 1 on
// a GPU with up to about 240 SMs (the per-block partial sums of y take
// SMs x d x 4 bytes; at most 10 MB on a 152-SM GB300). Every GPU that loads
// the library holds it until the process exits. All calls on a device share
// it: calls that can overlap on the GPU (different streams, or the same array
// used from two threads without ordering) race on it and must be serialized
// by the caller. No part of it needs clearing between calls: every scratch
// value the kernels read is written earlier in the same call.
#include <mutex>

#include "internal.h"

namespace sffn {

namespace {

constexpr size_t kStaticWsBytes = 16u << 20;  // 16 MiB

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
std::mutex g_ws_mutex;
void* g_ws_ptr[kMaxDevices] = {};

// Device address of g_static_ws on `dev` (the current device), looked up once
// per device. The host-side name g_static_ws is only a stand-in for the
// device symbol and must never be passed to a kernel.
sffn_status static_ws_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("sffn_decode_step_static_ws: device ordinal beyond the supported range");
    return SFFN_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return cuda_fail(e, "sffn_decode_step_static_ws: cudaGetSymbolAddress");
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return SFFN_OK;
}

}  // namespace

}  // namespace sffn

using namespace sffn;

extern "C" sffn_status sffn_decode_step_static_ws(const sffn_layer* L, const float* x, int32_t B, float thres,
                                                  const sffn_masks* m, float* y, float* x_out,
                                                  sffn_stream stream) {
  if (!L) {
    set_error("sffn_decode_step_static_ws: layer is NULL");
    return SFFN_ERR_INVALID_ARG;
  }
  if (!x || (reinterpret_cast<uintptr_t>(x) & 15)) {
    set_error("sffn_decode_step_static_ws: x must be a non-NULL 16-byte aligned device pointer");
    return SFFN_ERR_INVALID_ARG;
  }
  if (!m || !m->nmask) {
    set_error("sffn_decode_step_static_ws: masks and masks->nmask are required");
    return SFFN_ERR_INVALID_ARG;
  }
  if (!y || (reinterpret_cast<uintptr_t>(y) & 15) || y == x) {
    set_error("sffn_decode_step_static_ws: y must be a 16-byte aligned device pointer that differs from x");
    return SFFN_ERR_INVALID_ARG;
  }
  if (x_out && (x_out == y || (reinterpret_cast<uintptr_t>(x_out) & 15))) {
    set_error("sffn_decode_step_static_ws: x_out must be 16-byte aligned and differ from y");
    return SFFN_ERR_INVALID_ARG;
  }
  if (B < 1 || B > L->desc.max_batch) {
    set_error("sffn_decode_step_static_ws: B must be in [1, max_batch]");
    return SFFN_ERR_INVALID_ARG;
  }
  if (B > 1) {
    set_error("sffn_decode_step_static_ws: batch sizes above 1 are not implemented in this build");
    return SFFN_ERR_UNSUPPORTED;
  }
  const WsLayout w = ws_layout(*L, B);
  if (w.total > kStaticWsBytes) {
    set_error("sffn_decode_step_static_ws: this layer needs more scratch than the 16 MiB static array holds; "
              "use sffn_decode_step with a caller workspace");
    return SFFN_ERR_INVALID_ARG;
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "sffn_decode_step_static_ws: cudaGetDevice");
  if (dev != L->device) {
    set_error("sffn_decode_step_static_ws: the current CUDA device is not the one the layer was created on");
    return SFFN_ERR_INVALID_ARG;
  }
  void* ws = nullptr;
  sffn_status rc = static_ws_address(dev, &ws);
  if (rc != SFFN_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  char* base = static_cast<char*>(ws);
  float* hid = reinterpret_cast<float*>(base + w.hid);
  float* part = reinterpret_cast<float*>(base + w.partials);
  int32_t* kept = reinterpret_cast<int32_t*>(base + w.kept);
  e = launch_pred_hidden(*L, x, hid, st);
  if (e == cudaSuccess) e = launch_pred_scores(*L, hid, thres, m->nmask, st);
  if (e == cudaSuccess) e = launch_ffn(*L, x, m->nmask, m->idx, m->count, m->gmask, part, kept, st);
  if (e == cudaSuccess) e = launch_ffn_reduce(*L, part, kept, x, y, x_out, st);
  if (e != cudaSuccess) return cuda_fail(e, "sffn_decode_step_static_ws: launch");
  return SFFN_OK;
}
