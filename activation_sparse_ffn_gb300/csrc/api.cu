// The extern "C" entry points of libsffn.so: argument checks, handles,
// workspace layout and the order in which the kernels are enqueued.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "internal.h"

namespace sffn {

namespace {
thread_local std::string g_last_error;

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int wbytes_of(int wdtype) { return wdtype == SFFN_F32 ? 4 : 2; }

sffn_status invalid(const char* msg) {
  set_error(msg);
  return SFFN_ERR_INVALID_ARG;
}

sffn_status check_device(int want) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != want) return invalid("the current CUDA device is not the one the handle was created on");
  return SFFN_OK;
}

// Largest batch the automatic choice gives to the CUDA-core arm: on GB300 it
// beats the tensor-core products at B = 2 and loses from B = 3 on (Falcon-40B-
// shaped layer: 63.4 against 67.2 us at B = 2, 79.7 against 70.9 at B = 3).
constexpr int kAutoCudaCoreMaxBatch = 2;

// Whether a batched call on this layer runs the CUDA-core arm (batch_cc.cu)
// rather than the tensor-core products (batch.cu).
bool use_cuda_cores(const sffn_layer& L, int B) {
  if (L.batch_path == SFFN_BATCH_CUDA_CORES) return B <= kCcMaxBatch;
  if (L.batch_path == SFFN_BATCH_AUTO && B <= kAutoCudaCoreMaxBatch) {
    std::string why;
    return batch_cc_supported(L, B, &why);
  }
  return false;
}

size_t ws_bytes_for(const sffn_layer& L, int B) {
  if (B == 1) return ws_layout(L, 1).total;
  // either arm may serve the call (sffn_layer_set_batch_path can change between calls)
  const size_t tc = batch_ws_layout(L, B).total;
  const size_t cc = B <= kCcMaxBatch ? batch_cc_ws_layout(L, B).total : 0;
  return std::max(tc, cc);
}

sffn_status check_ws(const sffn_layer* L, int B, const void* ws, size_t ws_bytes) {
  if (!ws) return invalid("ws is NULL");
  if (!aligned(ws, 256)) return invalid("ws must be 256-byte aligned");
  if (ws_bytes < ws_bytes_for(*L, B)) return invalid("ws_bytes is smaller than sffn_workspace_bytes(layer, B)");
  return SFFN_OK;
}

sffn_status check_batch(const sffn_layer* L, int B) {
  if (B < 1 || B > L->desc.max_batch) return invalid("B must be in [1, max_batch]");
  std::string why;
  if (B > 1 && !(use_cuda_cores(*L, B) ? batch_cc_supported(*L, B, &why) : batch_supported(*L, &why))) {
    set_error(why);
    return SFFN_ERR_UNSUPPORTED;
  }
  return SFFN_OK;
}

cudaError_t launch_batched(const sffn_layer& L, const float* x, int B, float thres, const sffn_masks* m,
                           bool predict, bool forward, float* y, float* x_out, void* ws, cudaStream_t st) {
  if (use_cuda_cores(L, B)) return launch_batch_cc(L, x, B, thres, m, predict, forward, y, x_out, ws, st);
  return launch_batch(L, x, B, thres, m, predict, forward, y, x_out, ws, st);
}

// Records the layer's trace event for kernel slot k (if any) around `launch`.
template <typename F>
cudaError_t traced(const sffn_layer& L, int k, cudaStream_t st, F&& launch) {
  cudaError_t e = cudaSuccess;
  if (L.trace_begin[k]) e = cudaEventRecord(L.trace_begin[k], st);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess && L.trace_end[k]) e = cudaEventRecord(L.trace_end[k], st);
  return e;
}

}  // namespace

void set_error(const std::string& msg) { g_last_error = msg; }

sffn_status cuda_fail(cudaError_t e, const char* what) {
  char buf[512];
  snprintf(buf, sizeof(buf), "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  g_last_error = buf;
  if (e == cudaErrorMemoryAllocation) return SFFN_ERR_OOM;
  return SFFN_ERR_CUDA;
}

WsLayout ws_layout(const sffn_layer& L, int B) {
  WsLayout w;
  size_t off = 0;
  w.hid = off;
  off = align256(off + (size_t)B * L.desc.h * 4);
  w.partials = off;
  off = align256(off + (size_t)B * ffn_blocks(L) * L.desc.d * 4);
  w.kept = off;
  off = align256(off + (size_t)ffn_blocks(L) * 4);
  w.total = off;
  return w;
}

}  // namespace sffn

using namespace sffn;

extern "C" {

const char* sffn_status_string(sffn_status s) {
  switch (s) {
    case SFFN_OK: return "SFFN_OK";
    case SFFN_ERR_INVALID_ARG: return "SFFN_ERR_INVALID_ARG";
    case SFFN_ERR_UNSUPPORTED: return "SFFN_ERR_UNSUPPORTED";
    case SFFN_ERR_CUDA: return "SFFN_ERR_CUDA";
    case SFFN_ERR_TIMEOUT: return "SFFN_ERR_TIMEOUT";
    case SFFN_ERR_OOM: return "SFFN_ERR_OOM";
    case SFFN_ERR_DEVICE: return "SFFN_ERR_DEVICE";
  }
  return "SFFN_ERR_UNKNOWN";
}

const char* sffn_last_error(void) { return g_last_error.c_str(); }

const char* sffn_version(void) { return "sffn 0.1 sm_103a"; }

sffn_status sffn_layer_validate(const sffn_layer_desc* desc) {
  if (!desc) return invalid("desc is NULL");
  const sffn_layer_desc& D = *desc;
  if (D.wdtype != SFFN_F32 && D.wdtype != SFFN_F16 && D.wdtype != SFFN_BF16) return invalid("wdtype is not an sffn_dtype");
  if (D.act != SFFN_ACT_RELU && D.act != SFFN_ACT_REGLU && D.act != SFFN_ACT_SWIGLU && D.act != SFFN_ACT_RELU2)
    return invalid("act is not an sffn_act");
  if (D.d < 8 || D.d > 16384 || D.d % 8) return invalid("d must be a multiple of 8 in [8, 16384]");
  if ((long long)D.d * wbytes_of(D.wdtype) > 32768) return invalid("a weight row (d * element size) must be at most 32 KB");
  if (D.h < 8 || D.h % 8) return invalid("h must be a positive multiple of 8");
  if ((long long)D.h * wbytes_of(D.wdtype) > 2048) return invalid("a predictor row (h * element size) must be at most 2 KB");
  if (D.group_size != 32 && D.group_size != 64) return invalid("group_size must be 32 or 64");
  if (D.f < D.group_size || D.f % D.group_size) return invalid("f must be a positive multiple of group_size");
  if (D.f / D.group_size > 1024) return invalid("at most 1024 groups per layer");
  if (D.max_batch < 1 || D.max_batch > 32) return invalid("max_batch must be in [1, 32]");
  if (D.ffn_format != SFFN_FFN_ROWS && D.ffn_format != SFFN_FFN_Q8 && D.ffn_format != SFFN_FFN_Q4)
    return invalid("ffn_format is not an sffn_ffn_format");
  if (D.ffn_format == SFFN_FFN_Q8 && (D.wdtype == SFFN_F32 || D.d % 16))
    return invalid("8-bit FFN rows need a 16-bit predictor (wdtype fp16 or bf16) and d a multiple of 16");
  if (D.ffn_format == SFFN_FFN_Q4 && (D.wdtype == SFFN_F32 || D.d % 32))
    return invalid("4-bit FFN rows need a 16-bit predictor (wdtype fp16 or bf16) and d a multiple of 32");
  return SFFN_OK;
}

sffn_status sffn_layer_create(const sffn_layer_desc* desc, sffn_layer** out) {
  if (!out) return invalid("out is NULL");
  sffn_status rc = sffn_layer_validate(desc);
  if (rc != SFFN_OK) return rc;
  sffn_layer* L = new (std::nothrow) sffn_layer();
  if (!L) return invalid("host allocation failed");
  L->desc = *desc;
  L->wbytes = wbytes_of(desc->wdtype);
  L->fbits = desc->ffn_format == SFFN_FFN_Q8 ? 8 : desc->ffn_format == SFFN_FFN_Q4 ? 4 : 8 * L->wbytes;
  L->n_groups = desc->f / desc->group_size;
  L->nwords = desc->f / 32;
  L->gwords = (L->n_groups + 31) / 32;
  cudaError_t e = cudaGetDevice(&L->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&L->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, L->device);
  if (e != cudaSuccess) {
    delete L;
    return cuda_fail(e, "sffn_layer_create: device query");
  }
  L->score_stages = score_stages_for(*L);
  L->ffn_stages = ffn_stages_for(*L);
  if (L->ffn_stages < 2) {
    delete L;
    set_error("sffn_layer_create: the FFN ring does not fit in shared memory for this shape");
    return SFFN_ERR_UNSUPPORTED;
  }
  const size_t d = desc->d, f = desc->f, h = desc->h, wb = L->wbytes, frow = ffn_row_bytes(*L);
  const bool q8 = desc->ffn_format != SFFN_FFN_ROWS;  // scaled codes (8-bit or 4-bit)
  struct {
    void** p;
    size_t bytes;
  } allocs[] = {
      {&L->W1, h * d * wb},
      {(void**)&L->b1, h * 4},
      {&L->W2, f * h * wb},
      {(void**)&L->b2, f * 4},
      {&L->up, f * frow},
      {&L->gate, act_gated(desc->act) ? f * frow : 0},
      {&L->downT, f * frow},
      {(void**)&L->up_s, q8 ? f * 4 : 0},
      {(void**)&L->gate_s, q8 && act_gated(desc->act) ? f * 4 : 0},
      {(void**)&L->down_s, q8 ? f * 4 : 0},
      {(void**)&L->perm, f * 4},
      {(void**)&L->err, 256},
  };
  for (auto& a : allocs) {
    if (!a.bytes) continue;
    e = cudaMalloc(a.p, a.bytes);
    if (e != cudaSuccess) {
      rc = cuda_fail(e, "sffn_layer_create: cudaMalloc");
      sffn_layer_destroy(L);
      return rc;
    }
  }
  e = cudaMemset(L->err, 0, 256);
  if (e == cudaSuccess) e = configure_kernels(*L);
  if (e == cudaSuccess) e = configure_predict_kernels(*L);
  if (e == cudaSuccess) e = configure_batch_kernels(*L);
  if (e == cudaSuccess) e = configure_batch_cc_kernels(*L);
  if (e != cudaSuccess) {
    rc = cuda_fail(e, "sffn_layer_create: kernel set-up");
    sffn_layer_destroy(L);
    return rc;
  }
  *out = L;
  return SFFN_OK;
}

sffn_status sffn_layer_pack(sffn_layer* L, const void* W1, const float* b1, const void* W2, const float* b2,
                            const void* up, const void* gate, const void* down, const int32_t* perm,
                            sffn_stream stream) {
  if (!L) return invalid("layer is NULL");
  if (L->desc.ffn_format == SFFN_FFN_Q8) return invalid("this layer stores 8-bit FFN rows: use sffn_layer_pack_q8");
  if (L->desc.ffn_format == SFFN_FFN_Q4) return invalid("this layer stores 4-bit FFN rows: use sffn_layer_pack_q4");
  if (!W1 || !W2 || !up || !down) return invalid("W1, W2, up and down are required");
  if (act_gated(L->desc.act) && !gate) return invalid("gate is required for ReGLU and SwiGLU");
  const void* ptrs[] = {W1, W2, up, down, gate, b1, b2, perm};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return invalid("weight, bias and perm pointers must be 16-byte aligned");
  sffn_status rc = check_device(L->device);
  if (rc != SFFN_OK) return rc;
  return pack_layer(*L, W1, b1, W2, b2, up, act_gated(L->desc.act) ? gate : nullptr, down, perm,
                    (cudaStream_t)stream);
}

namespace {

sffn_status pack_codes(sffn_layer* L, const void* W1, const float* b1, const void* W2, const float* b2,
                       const int8_t* up_q, const float* up_scale, const int8_t* gate_q, const float* gate_scale,
                       const int8_t* down_q, const float* down_scale, const int32_t* perm, sffn_stream stream) {
  if (!W1 || !W2 || !up_q || !up_scale || !down_q || !down_scale)
    return invalid("W1, W2, up_q, up_scale, down_q and down_scale are required");
  const bool gated = act_gated(L->desc.act);
  if (gated && (!gate_q || !gate_scale)) return invalid("gate_q and gate_scale are required for ReGLU and SwiGLU");
  const void* ptrs[] = {W1, W2, up_q, up_scale, down_q, down_scale, gate_q, gate_scale, b1, b2, perm};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return invalid("weight, scale, bias and perm pointers must be 16-byte aligned");
  sffn_status rc = check_device(L->device);
  if (rc != SFFN_OK) return rc;
  return pack_layer(*L, W1, b1, W2, b2, up_q, gated ? gate_q : nullptr, down_q, perm, (cudaStream_t)stream,
                    up_scale, gated ? gate_scale : nullptr, down_scale);
}

}  // namespace

sffn_status sffn_layer_pack_q8(sffn_layer* L, const void* W1, const float* b1, const void* W2, const float* b2,
                               const int8_t* up_q, const float* up_scale, const int8_t* gate_q,
                               const float* gate_scale, const int8_t* down_q, const float* down_scale,
                               const int32_t* perm, sffn_stream stream) {
  if (!L) return invalid("layer is NULL");
  if (L->desc.ffn_format != SFFN_FFN_Q8) return invalid("sffn_layer_pack_q8 needs a layer with ffn_format SFFN_FFN_Q8");
  return pack_codes(L, W1, b1, W2, b2, up_q, up_scale, gate_q, gate_scale, down_q, down_scale, perm, stream);
}

sffn_status sffn_layer_pack_q4(sffn_layer* L, const void* W1, const float* b1, const void* W2, const float* b2,
                               const int8_t* up_q, const float* up_scale, const int8_t* gate_q,
                               const float* gate_scale, const int8_t* down_q, const float* down_scale,
                               const int32_t* perm, sffn_stream stream) {
  if (!L) return invalid("layer is NULL");
  if (L->desc.ffn_format != SFFN_FFN_Q4) return invalid("sffn_layer_pack_q4 needs a layer with ffn_format SFFN_FFN_Q4");
  return pack_codes(L, W1, b1, W2, b2, up_q, up_scale, gate_q, gate_scale, down_q, down_scale, perm, stream);
}

sffn_status sffn_layer_get_desc(const sffn_layer* L, sffn_layer_desc* out) {
  if (!L || !out) return invalid("layer or out is NULL");
  *out = L->desc;
  return SFFN_OK;
}

sffn_status sffn_layer_packed(const sffn_layer* L, sffn_packed_view* out) {
  if (!L || !out) return invalid("layer or out is NULL");
  out->W1 = L->W1;
  out->b1 = L->b1;
  out->W2 = L->W2;
  out->b2 = L->b2;
  out->up = L->up;
  out->gate = L->gate;
  out->downT = L->downT;
  out->perm = L->perm;
  out->up_scale = L->up_s;
  out->gate_scale = L->gate_s;
  out->down_scale = L->down_s;
  return SFFN_OK;
}

sffn_status sffn_layer_set_trace(sffn_layer* L, const sffn_trace* t) {
  if (!L) return invalid("layer is NULL");
  for (int k = 0; k < 4; ++k) {
    L->trace_begin[k] = t ? static_cast<cudaEvent_t>(t->begin[k]) : nullptr;
    L->trace_end[k] = t ? static_cast<cudaEvent_t>(t->end[k]) : nullptr;
  }
  return SFFN_OK;
}

sffn_status sffn_layer_set_grid(sffn_layer* L, int32_t ffn_blocks, int32_t score_blocks) {
  if (!L) return invalid("layer is NULL");
  if (ffn_blocks < 0 || ffn_blocks > L->num_sms || score_blocks < 0 || score_blocks > L->num_sms)
    return invalid("sffn_layer_set_grid: block counts must lie in [0, number of SMs]");
  const int old_ffn = L->ffn_grid, old_stages = L->ffn_stages;
  L->ffn_grid = ffn_blocks;
  L->ffn_stages = ffn_stages_for(*L);  // the per-block neuron list grows as blocks get fewer
  if (L->ffn_stages < 2 || ffn_smem(*L) + 1024 > (size_t)L->smem_optin) {
    L->ffn_grid = old_ffn;
    L->ffn_stages = old_stages;
    return invalid("sffn_layer_set_grid: too few FFN blocks for this layer's shared-memory ring");
  }
  L->score_grid = score_blocks;
  return SFFN_OK;
}

sffn_status sffn_layer_set_batch_path(sffn_layer* L, int32_t path) {
  if (!L) return invalid("layer is NULL");
  if (path != SFFN_BATCH_AUTO && path != SFFN_BATCH_TENSOR && path != SFFN_BATCH_CUDA_CORES)
    return invalid("path is not an sffn_batch_path");
  L->batch_path = path;
  return SFFN_OK;
}

int32_t sffn_layer_batch_arm(const sffn_layer* L, int32_t B) {
  if (!L || B < 2 || B > L->desc.max_batch) return -1;
  std::string why;
  if (use_cuda_cores(*L, B)) return batch_cc_supported(*L, B, &why) ? SFFN_BATCH_CUDA_CORES : -1;
  return batch_supported(*L, &why) ? SFFN_BATCH_TENSOR : -1;
}

sffn_status sffn_layer_set_zero_skip(sffn_layer* L, int32_t enable, int32_t* rows_read) {
  if (!L) return invalid("layer is NULL");
  if (rows_read && !aligned(rows_read, 4)) return invalid("rows_read must be 4-byte aligned");
  L->zero_skip = enable != 0;
  L->rows_read = enable ? rows_read : nullptr;
  return SFFN_OK;
}

sffn_status sffn_layer_set_l2_resident(sffn_layer* L, const uint32_t* resident) {
  if (!L) return invalid("layer is NULL");
  if (resident && (reinterpret_cast<uintptr_t>(resident) & 3)) return invalid("resident must be 4-byte aligned");
  L->l2_resident = resident;
  return SFFN_OK;
}

sffn_status sffn_layer_set_next(sffn_layer* L, const sffn_layer* next) {
  if (!L) return invalid("layer is NULL");
  if (next && next->device != L->device) return invalid("sffn_layer_set_next: next lives on another device");
  L->next = next;
  return SFFN_OK;
}

size_t sffn_workspace_bytes(const sffn_layer* L, int32_t B) {
  if (!L || B < 1 || B > L->desc.max_batch) return 0;
  return ws_bytes_for(*L, B);
}

static sffn_status read_error_word(uint32_t* err, cudaStream_t st) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "check_error: synchronize");
  uint32_t h = 0;
  e = cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && h) e = cudaMemset(err, 0, 4);
  if (e != cudaSuccess) return cuda_fail(e, "check_error: read error word");
  if (h == SFFN_ERR_TIMEOUT) {
    set_error("a bounded device-side wait ran out");
    return SFFN_ERR_TIMEOUT;
  }
  if (h) {
    set_error("the device flagged bad data");
    return SFFN_ERR_DEVICE;
  }
  return SFFN_OK;
}

sffn_status sffn_layer_check_error(const sffn_layer* L, sffn_stream stream) {
  if (!L) return invalid("layer is NULL");
  return read_error_word(L->err, (cudaStream_t)stream);
}

void sffn_layer_destroy(sffn_layer* L) {
  if (!L) return;
  void* ps[] = {L->W1, L->b1, L->W2, L->b2, L->up, L->gate, L->downT, L->perm, L->up_s, L->gate_s, L->down_s, L->err};
  for (void* p : ps)
    if (p) cudaFree(p);
  delete L;
}

// ---------------------------------------------------------------- hot calls

static sffn_status check_hot(const sffn_layer* L, const float* x, int B, const sffn_masks* m, const void* ws,
                             size_t ws_bytes) {
  if (!L) return invalid("layer is NULL");
  if (!x || !aligned(x, 16)) return invalid("x must be a non-NULL 16-byte aligned device pointer");
  if (!m || !m->nmask) return invalid("masks and masks->nmask are required");
  sffn_status rc = check_batch(L, B);
  if (rc != SFFN_OK) return rc;
  rc = check_ws(L, B, ws, ws_bytes);
  if (rc != SFFN_OK) return rc;
  return check_device(L->device);
}

sffn_status sffn_predict(const sffn_layer* L, const float* x, int32_t B, float thres, const sffn_masks* m, void* ws,
                         size_t ws_bytes, sffn_stream stream) {
  sffn_status rc = check_hot(L, x, B, m, ws, ws_bytes);
  if (rc != SFFN_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (B > 1) {
    cudaError_t e = launch_batched(*L, x, B, thres, m, true, false, nullptr, nullptr, ws, st);
    if (e != cudaSuccess) return cuda_fail(e, "sffn_predict: launch");
    return SFFN_OK;
  }
  const WsLayout w = ws_layout(*L, B);
  float* hid = reinterpret_cast<float*>(static_cast<char*>(ws) + w.hid);
  cudaError_t e = traced(*L, 0, st, [&] { return launch_pred_hidden(*L, x, hid, st); });
  if (e == cudaSuccess) e = traced(*L, 1, st, [&] { return launch_pred_scores(*L, hid, thres, m->nmask, st); });
  if (e == cudaSuccess && (m->idx || m->count || m->gmask))
    e = launch_mask_views(*L, m->nmask, m->idx, m->count, m->gmask, st);
  if (e != cudaSuccess) return cuda_fail(e, "sffn_predict: launch");
  return SFFN_OK;
}

sffn_status sffn_forward(const sffn_layer* L, const float* x, int32_t B, const sffn_masks* m, float* y,
                         float* x_out, void* ws, size_t ws_bytes, sffn_stream stream) {
  sffn_status rc = check_hot(L, x, B, m, ws, ws_bytes);
  if (rc != SFFN_OK) return rc;
  if (!y || !aligned(y, 16)) return invalid("y must be a non-NULL 16-byte aligned device pointer");
  if (y == x) return invalid("y must not alias x");
  if (x_out && (x_out == y || !aligned(x_out, 16))) return invalid("x_out must be 16-byte aligned and differ from y");
  cudaStream_t st = (cudaStream_t)stream;
  if (B > 1) {
    cudaError_t e = launch_batched(*L, x, B, 0.f, m, false, true, y, x_out, ws, st);
    if (e != cudaSuccess) return cuda_fail(e, "sffn_forward: launch");
    return SFFN_OK;
  }
  const WsLayout w = ws_layout(*L, B);
  char* base = static_cast<char*>(ws);
  float* part = reinterpret_cast<float*>(base + w.partials);
  int32_t* kept = reinterpret_cast<int32_t*>(base + w.kept);
  cudaError_t e =
      traced(*L, 2, st, [&] { return launch_ffn(*L, x, m->nmask, nullptr, nullptr, nullptr, part, kept, st); });
  if (e == cudaSuccess) e = traced(*L, 3, st, [&] { return launch_ffn_reduce(*L, part, kept, x, y, x_out, st); });
  if (e != cudaSuccess) return cuda_fail(e, "sffn_forward: launch");
  return SFFN_OK;
}

static sffn_status check_step(const sffn_layer* L, const float* x, int B, const sffn_masks* m, float* y,
                              float* x_out, const void* ws, size_t ws_bytes) {
  sffn_status rc = check_hot(L, x, B, m, ws, ws_bytes);
  if (rc != SFFN_OK) return rc;
  if (!y || !aligned(y, 16)) return invalid("y must be a non-NULL 16-byte aligned device pointer");
  if (y == x) return invalid("y must not alias x");
  if (x_out && (x_out == y || !aligned(x_out, 16))) return invalid("x_out must be 16-byte aligned and differ from y");
  return SFFN_OK;
}

// predict + forward of one layer (arguments already checked)
static sffn_status decode_step_launch(const sffn_layer* L, const float* x, int32_t B, float thres,
                                      const sffn_masks* m, float* y, float* x_out, void* ws, cudaStream_t st) {
  if (B > 1) {
    cudaError_t e = launch_batched(*L, x, B, thres, m, true, true, y, x_out, ws, st);
    if (e != cudaSuccess) return cuda_fail(e, "sffn_decode_step: launch");
    return SFFN_OK;
  }
  const WsLayout w = ws_layout(*L, B);
  char* base = static_cast<char*>(ws);
  float* hid = reinterpret_cast<float*>(base + w.hid);
  float* part = reinterpret_cast<float*>(base + w.partials);
  int32_t* kept = reinterpret_cast<int32_t*>(base + w.kept);
  cudaError_t e = traced(*L, 0, st, [&] { return launch_pred_hidden(*L, x, hid, st); });
  if (e == cudaSuccess) e = traced(*L, 1, st, [&] { return launch_pred_scores(*L, hid, thres, m->nmask, st); });
  if (e == cudaSuccess)
    e = traced(*L, 2, st, [&] {
      return launch_ffn(*L, x, m->nmask, m->idx, m->count, m->gmask, part, kept, st);
    });
  if (e == cudaSuccess) e = traced(*L, 3, st, [&] { return launch_ffn_reduce(*L, part, kept, x, y, x_out, st); });
  if (e != cudaSuccess) return cuda_fail(e, "sffn_decode_step: launch");
  return SFFN_OK;
}

sffn_status sffn_decode_step(const sffn_layer* L, const float* x, int32_t B, float thres, const sffn_masks* m,
                             float* y, float* x_out, void* ws, size_t ws_bytes, sffn_stream stream) {
  sffn_status rc = check_step(L, x, B, m, y, x_out, ws, ws_bytes);
  if (rc != SFFN_OK) return rc;
  return decode_step_launch(L, x, B, thres, m, y, x_out, ws, (cudaStream_t)stream);
}

static sffn_status check_tam_args(const tam_state* S, int32_t layer0, int32_t n_layers, float lambda, float eps,
                                  int32_t K) {
  if (!S) return invalid("tam is NULL");
  if (layer0 < 0 || n_layers < 1 || layer0 + n_layers > S->n_layers) return invalid("layer range out of bounds");
  if (!(lambda < 1.f) || std::isnan(lambda)) return invalid("lambda must be < 1 (negative: use the state's lambda)");
  if (!(eps >= 0.f) || std::isinf(eps)) return invalid("eps must be finite and >= 0");
  if (K < 0 || K > S->n_groups) return invalid("capacity_k must be in [0, n_groups]");
  return SFFN_OK;
}

sffn_status sffn_decode_step_tam(const sffn_layer* L, tam_state* S, int32_t layer, const float* x, int32_t B,
                                 float thres, const sffn_masks* m, float* y, float* x_out, void* ws, size_t ws_bytes,
                                 float lambda, float eps, int32_t K, const tam_outputs* out, sffn_stream stream) {
  sffn_status rc = check_step(L, x, B, m, y, x_out, ws, ws_bytes);
  if (rc != SFFN_OK) return rc;
  rc = check_tam_args(S, layer, 1, lambda, eps, K);
  if (rc != SFFN_OK) return rc;
  if (S->n_groups != L->n_groups) return invalid("the momentum state's group count differs from the layer's");
  if (S->device != L->device) return invalid("the momentum state lives on another device");
  // the momentum step reads the token's group bitmask (B = 1) or the batch union's
  uint32_t* gm = B == 1 ? m->gmask : m->ugmask;
  if (!gm || !aligned(gm, 4))
    return invalid(B == 1 ? "masks->gmask is required (the momentum step reads it)"
                          : "masks->ugmask is required (the momentum step reads the union group bitmask)");
  cudaStream_t st = (cudaStream_t)stream;
  rc = decode_step_launch(L, x, B, thres, m, y, x_out, ws, st);
  if (rc != SFFN_OK) return rc;
  tam_outputs o = {};
  if (out) o = *out;
  cudaError_t e = launch_tam_update(*S, layer, 1, gm, L->gwords, lambda, eps, K, o, st);
  if (e != cudaSuccess) return cuda_fail(e, "sffn_decode_step_tam: launch");
  return SFFN_OK;
}

// ---------------------------------------------------------------- TAM

sffn_status tam_create(int32_t n_layers, int32_t n_groups, float lambda0, tam_state** out) {
  if (!out) return invalid("out is NULL");
  if (n_layers < 1 || n_layers > 4096) return invalid("n_layers must be in [1, 4096]");
  if (n_groups < 1 || n_groups > 1024) return invalid("n_groups must be in [1, 1024]");
  if (!(lambda0 > 0.f && lambda0 < 1.f)) return invalid("lambda0 must be in (0, 1)");
  tam_state* S = new (std::nothrow) tam_state();
  if (!S) return invalid("host allocation failed");
  S->n_layers = n_layers;
  S->n_groups = n_groups;
  S->gwords = (n_groups + 31) / 32;
  cudaError_t e = cudaGetDevice(&S->device);
  if (e == cudaSuccess) e = cudaMalloc(&S->scores, (size_t)n_layers * n_groups * 4);
  if (e == cudaSuccess) e = cudaMalloc(&S->lambdas, (size_t)n_layers * 4);
  if (e == cudaSuccess) e = cudaMalloc(&S->resident, (size_t)n_layers * S->gwords * 4);
  if (e == cudaSuccess) e = cudaMalloc(&S->err, 256);
  if (e == cudaSuccess) e = cudaMemset(S->scores, 0, (size_t)n_layers * n_groups * 4);
  if (e == cudaSuccess) e = cudaMemset(S->resident, 0, (size_t)n_layers * S->gwords * 4);
  if (e == cudaSuccess) e = cudaMemset(S->err, 0, 256);
  if (e == cudaSuccess) {
    float* h = new (std::nothrow) float[n_layers];
    if (!h) {
      tam_destroy(S);
      return invalid("host allocation failed");
    }
    for (int i = 0; i < n_layers; ++i) h[i] = lambda0;
    e = cudaMemcpy(S->lambdas, h, (size_t)n_layers * 4, cudaMemcpyHostToDevice);
    delete[] h;
  }
  if (e != cudaSuccess) {
    sffn_status rc = cuda_fail(e, "tam_create");
    tam_destroy(S);
    return rc;
  }
  *out = S;
  return SFFN_OK;
}

sffn_status tam_update(tam_state* S, int32_t layer0, int32_t n_layers, const uint32_t* gmask, int32_t gstride,
                       float lambda, float eps, int32_t K, const tam_outputs* out, sffn_stream stream) {
  sffn_status rc = check_tam_args(S, layer0, n_layers, lambda, eps, K);
  if (rc != SFFN_OK) return rc;
  if (!gmask || !aligned(gmask, 4)) return invalid("gmask must be a non-NULL 4-byte aligned device pointer");
  if (gstride < S->gwords) return invalid("gmask_stride is shorter than a group bitset");
  rc = check_device(S->device);
  if (rc != SFFN_OK) return rc;
  tam_outputs o = {};
  if (out) o = *out;
  cudaError_t e = launch_tam_update(*S, layer0, n_layers, gmask, gstride, lambda, eps, K, o, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "tam_update: launch");
  return SFFN_OK;
}

sffn_status tam_adapt(tam_state* S, int32_t layer0, int32_t n_layers, const uint8_t* stall, float alpha, float lo,
                      float hi, sffn_stream stream) {
  if (!S) return invalid("tam is NULL");
  if (layer0 < 0 || n_layers < 1 || layer0 + n_layers > S->n_layers) return invalid("layer range out of bounds");
  if (!stall) return invalid("stall is NULL");
  if (!(alpha >= 0.f) || std::isinf(alpha)) return invalid("alpha must be finite and >= 0");
  if (!(lo > 0.f && lo <= hi && hi < 1.f)) return invalid("need 0 < lo <= hi < 1");
  sffn_status rc = check_device(S->device);
  if (rc != SFFN_OK) return rc;
  cudaError_t e = launch_tam_adapt(*S, layer0, n_layers, stall, alpha, lo, hi, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "tam_adapt: launch");
  return SFFN_OK;
}

sffn_status tam_get_state(const tam_state* S, float* scores, float* lambdas, uint32_t* resident, sffn_stream stream) {
  if (!S) return invalid("tam is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (scores) e = cudaMemcpyAsync(scores, S->scores, (size_t)S->n_layers * S->n_groups * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && lambdas)
    e = cudaMemcpyAsync(lambdas, S->lambdas, (size_t)S->n_layers * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && resident)
    e = cudaMemcpyAsync(resident, S->resident, (size_t)S->n_layers * S->gwords * 4, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "tam_get_state");
  return SFFN_OK;
}

sffn_status tam_set_state(tam_state* S, const float* scores, const float* lambdas, const uint32_t* resident,
                          sffn_stream stream) {
  if (!S) return invalid("tam is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (scores) e = cudaMemcpyAsync(S->scores, scores, (size_t)S->n_layers * S->n_groups * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && lambdas)
    e = cudaMemcpyAsync(S->lambdas, lambdas, (size_t)S->n_layers * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && resident)
    e = cudaMemcpyAsync(S->resident, resident, (size_t)S->n_layers * S->gwords * 4, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "tam_set_state");
  return SFFN_OK;
}

sffn_status tam_get_shape(const tam_state* S, int32_t* n_layers, int32_t* n_groups) {
  if (!S || !n_layers || !n_groups) return invalid("tam, n_layers or n_groups is NULL");
  *n_layers = S->n_layers;
  *n_groups = S->n_groups;
  return SFFN_OK;
}

sffn_status tam_check_error(const tam_state* S, sffn_stream stream) {
  if (!S) return invalid("tam is NULL");
  return read_error_word(S->err, (cudaStream_t)stream);
}

void tam_destroy(tam_state* S) {
  if (!S) return;
  void* ps[] = {S->scores, S->lambdas, S->resident, S->err};
  for (void* p : ps)
    if (p) cudaFree(p);
  delete S;
}

// ---------------------------------------------------------------- whole-stack decode

sffn_status sffn_stack_create(const sffn_layer* const* layers, int32_t n_layers, sffn_stack** out) {
  if (!out) return invalid("out is NULL");
  if (!layers) return invalid("layers is NULL");
  if (n_layers < 1 || n_layers > 4096) return invalid("n_layers must be in [1, 4096]");
  const sffn_layer* L0 = layers[0];
  if (!L0) return invalid("layers[0] is NULL");
  for (int l = 0; l < n_layers; ++l) {
    const sffn_layer* L = layers[l];
    if (!L) return invalid("a layer handle is NULL");
    const sffn_layer_desc &a = L->desc, &b = L0->desc;
    if (a.d != b.d || a.f != b.f || a.h != b.h || a.group_size != b.group_size || a.act != b.act ||
        a.wdtype != b.wdtype || a.ffn_format != b.ffn_format)
      return invalid("every layer of a stack must have the same shape, activation and storage");
    if (L->device != L0->device) return invalid("every layer of a stack must live on the same device");
  }
  std::string why;
  if (!stack_supported(*L0, &why)) {
    set_error(why);
    return SFFN_ERR_UNSUPPORTED;
  }
  sffn_status rc = check_device(L0->device);
  if (rc != SFFN_OK) return rc;
  sffn_stack* S = new (std::nothrow) sffn_stack();
  if (!S) return invalid("host allocation failed");
  S->n_layers = n_layers;
  S->device = L0->device;
  S->layers = new (std::nothrow) const sffn_layer*[n_layers];
  const size_t one = stack_layer_desc_bytes();
  unsigned char* table = new (std::nothrow) unsigned char[one * n_layers];
  if (!S->layers || !table) {
    delete[] table;
    sffn_stack_destroy(S);
    return invalid("host allocation failed");
  }
  for (int l = 0; l < n_layers; ++l) {
    S->layers[l] = layers[l];
    stack_fill_layer_desc(*layers[l], table + one * l);
  }
  cudaError_t e = cudaMalloc(&S->dev_layers, one * n_layers);
  if (e == cudaSuccess) e = cudaMalloc((void**)&S->bar, kStackBarBytes);
  if (e == cudaSuccess) e = cudaMalloc((void**)&S->err, 256);
  if (e == cudaSuccess) e = cudaMemcpy(S->dev_layers, table, one * n_layers, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(S->bar, 0, kStackBarBytes);
  if (e == cudaSuccess) e = cudaMemset(S->err, 0, 256);
  if (e == cudaSuccess) e = configure_stack_kernels(*L0);
  delete[] table;
  if (e != cudaSuccess) {
    rc = cuda_fail(e, "sffn_stack_create");
    sffn_stack_destroy(S);
    return rc;
  }
  *out = S;
  return SFFN_OK;
}

size_t sffn_stack_workspace_bytes(const sffn_stack* S) {
  if (!S) return 0;
  return stack_ws_bytes(*S->layers[0]);
}

sffn_status sffn_stack_decode(const sffn_stack* S, const float* x0, float* xs, float* ys, float thres,
                              const sffn_masks* m, void* ws, size_t ws_bytes, sffn_stream stream) {
  if (!S) return invalid("stack is NULL");
  const sffn_layer& L = *S->layers[0];
  const size_t d = (size_t)L.desc.d, nL = (size_t)S->n_layers;
  if (!x0 || !aligned(x0, 16)) return invalid("x0 must be a non-NULL 16-byte aligned device pointer");
  if (!xs || !aligned(xs, 16)) return invalid("xs must be a non-NULL 16-byte aligned device pointer");
  if (ys && !aligned(ys, 16)) return invalid("ys must be 16-byte aligned");
  if (!m || !m->nmask || !aligned(m->nmask, 4)) return invalid("masks and masks->nmask are required");
  // x0 may be one of xs's rows (the previous token's output), or lie apart from xs and ys
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x0), sa = reinterpret_cast<uintptr_t>(xs);
  const bool in_xs = xa >= sa && xa < sa + nL * d * 4;
  if (in_xs && (xa - sa) % (d * 4) != 0) return invalid("x0 inside xs must start one of its rows");
  if (ys) {
    const uintptr_t ya = reinterpret_cast<uintptr_t>(ys);
    if ((xa + d * 4 > ya && xa < ya + nL * d * 4) || (sa + nL * d * 4 > ya && sa < ya + nL * d * 4))
      return invalid("ys must not overlap x0 or xs");
  }
  if (!ws) return invalid("ws is NULL");
  if (!aligned(ws, 256)) return invalid("ws must be 256-byte aligned");
  if (ws_bytes < stack_ws_bytes(L)) return invalid("ws_bytes is smaller than sffn_stack_workspace_bytes(stack)");
  sffn_status rc = check_device(S->device);
  if (rc != SFFN_OK) return rc;
  cudaError_t e = launch_stack(*S, x0, xs, ys, thres, *m, ws, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "sffn_stack_decode: launch");
  return SFFN_OK;
}

sffn_status sffn_stack_check_error(const sffn_stack* S, sffn_stream stream) {
  if (!S) return invalid("stack is NULL");
  sffn_status rc = read_error_word(S->err, (cudaStream_t)stream);
  if (rc == SFFN_ERR_TIMEOUT || rc == SFFN_ERR_DEVICE) {
    // a kernel that wound down may have left the grid barrier half-way
    cudaError_t e = cudaMemset(S->bar, 0, kStackBarBytes);
    if (e != cudaSuccess) return cuda_fail(e, "sffn_stack_check_error: reset the grid barrier");
  }
  return rc;
}

void sffn_stack_destroy(sffn_stack* S) {
  if (!S) return;
  if (S->dev_layers) cudaFree(S->dev_layers);
  if (S->bar) cudaFree(S->bar);
  if (S->err) cudaFree(S->err);
  delete[] S->layers;
  delete S;
}

// ---------------------------------------------------------------- self-test

sffn_status sffn_selftest_wait_timeout(const sffn_layer* L, int32_t limit_us, sffn_stream stream) {
  if (!L) return invalid("layer is NULL");
  if (limit_us < 1 || limit_us > 100000) return invalid("limit_us must be in [1, 100000]");
  sffn_status rc = check_device(L->device);
  if (rc != SFFN_OK) return rc;
  cudaError_t e = launch_selftest_timeout(L->err, limit_us, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "sffn_selftest_wait_timeout: launch");
  return SFFN_OK;
}

}  // extern "C"
