// Host-side internals of libsffn: the layer and momentum-state handles, the
// workspace layout, and the per-kernel launchers implemented in the .cu files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

#include "sffn.h"

struct sffn_layer {
  sffn_layer_desc desc;
  int device = 0;
  int num_sms = 0;
  int smem_optin = 0;   // largest dynamic shared memory a block may request on this device
  // B = 1 grid sizes (sffn_layer_set_grid); 0 = one block per SM
  int ffn_grid = 0;
  int score_grid = 0;
  int wbytes = 0;       // bytes per stored predictor weight (and FFN weight unless quantized)
  int fbits = 0;        // bits per stored FFN weight (8 for SFFN_FFN_Q8, 4 for SFFN_FFN_Q4)
  int n_groups = 0;
  int nwords = 0;       // f / 32
  int gwords = 0;       // ceil(n_groups / 32)
  void* W1 = nullptr;
  float* b1 = nullptr;
  void* W2 = nullptr;
  float* b2 = nullptr;
  void* up = nullptr;
  void* gate = nullptr;
  void* downT = nullptr;
  int32_t* perm = nullptr;
  float* up_s = nullptr;     // SFFN_FFN_Q8 / Q4: per-slot row scales
  float* gate_s = nullptr;
  float* down_s = nullptr;
  uint32_t* err = nullptr;  // device error word
  bool has_b1 = false, has_b2 = false;
  // launch shapes chosen at create time
  int score_stages = 0;     // predictor-scores ring depth (one mask word per stage)
  int ffn_stages = 0;       // fused FFN ring depth (one neuron's up/gate rows, or as many downT rows)
  // optional L2 hint (sffn_layer_set_next): the layer whose predictor weights
  // this layer's FFN kernel prefetches
  const sffn_layer* next = nullptr;
  // optional hot-group set (sffn_layer_set_l2_resident): device bitset [gwords]
  const uint32_t* l2_resident = nullptr;
  // optional zero-skip (sffn_layer_set_zero_skip): downT rows only for h != 0,
  // and where to write how many were read (device, may be null)
  bool zero_skip = false;
  int32_t* rows_read = nullptr;
  // batched calls (sffn_layer_set_batch_path): SFFN_BATCH_AUTO, _TENSOR or _CUDA_CORES
  int batch_path = 0;
  // optional timing hooks (sffn_layer_set_trace)
  cudaEvent_t trace_begin[4] = {nullptr, nullptr, nullptr, nullptr};
  cudaEvent_t trace_end[4] = {nullptr, nullptr, nullptr, nullptr};
};

struct tam_state {
  int n_layers = 0;
  int n_groups = 0;
  int gwords = 0;
  int device = 0;
  float* scores = nullptr;     // [L][n_groups]
  float* lambdas = nullptr;    // [L]
  uint32_t* resident = nullptr;  // [L][gwords]
  uint32_t* err = nullptr;
};

// A stack of layers decoded by one persistent kernel per token
// (sffn_stack_decode). The layers are not owned.
struct sffn_stack {
  int n_layers = 0;
  int device = 0;
  const sffn_layer** layers = nullptr;  // host array [n_layers]
  void* dev_layers = nullptr;           // device table of the layers' packed arrays
  unsigned* bar = nullptr;              // grid barrier: arrival counter, generation
  uint32_t* err = nullptr;              // device error word
};

namespace sffn {

// Bytes of one stored FFN row (d weights).
inline size_t ffn_row_bytes(const sffn_layer& L) { return (size_t)L.desc.d * L.fbits / 8; }

// Whether an activation reads a gate row (ReGLU, SwiGLU) or not (ReLU, squared ReLU).
__host__ __device__ constexpr bool act_gated(int act) { return act == SFFN_ACT_REGLU || act == SFFN_ACT_SWIGLU; }

constexpr int kFfnSmemBudget = 224 * 1024;
constexpr int kFfnMaxStages = 12;
constexpr int kScoreSmemBudget = 192 * 1024;

// Workspace of one hot call for batch size B (offsets in bytes, 256-aligned).
struct WsLayout {
  size_t hid = 0;       // float [B][h]
  size_t partials = 0;  // float [B][ffn blocks][d]: per-block partial sums of y
  size_t kept = 0;      // int32 [ffn blocks]: downT rows each block read (zero-skip)
  size_t total = 0;
};
WsLayout ws_layout(const sffn_layer& L, int B);

// Workspace of a batched call (B > 1), offsets in bytes.
struct BatchWs {
  size_t xhl = 0, dh = 0, hidhl = 0, ds = 0, unmask = 0, uidx = 0, ucount = 0, dug = 0, hhl = 0, dy = 0, total = 0;
};
BatchWs batch_ws_layout(const sffn_layer& L, int B);
bool batch_supported(const sffn_layer& L, std::string* why);
// Per-token views and the union views of a batch (k_b_views); union_ready:
// the union words are already in unmask.
cudaError_t launch_batch_views(const sffn_layer& L, const sffn_masks* m, int B, uint32_t* unmask, int32_t* uidx,
                               int32_t* ucount, bool predict, bool union_ready, cudaStream_t st);

// CUDA-core arm of the batched step for 2..kCcMaxBatch tokens (batch_cc.cu).
constexpr int kCcMaxBatch = 4;
struct BatchCcWs {
  size_t hid = 0, unmask = 0, uidx = 0, ucount = 0, partials = 0, total = 0;
};
BatchCcWs batch_cc_ws_layout(const sffn_layer& L, int B);
bool batch_cc_supported(const sffn_layer& L, int B, std::string* why);
cudaError_t configure_batch_cc_kernels(const sffn_layer& L);
cudaError_t launch_batch_cc(const sffn_layer& L, const float* x, int B, float thres, const sffn_masks* m, bool predict,
                            bool forward, float* y, float* x_out, void* ws, cudaStream_t st);
cudaError_t configure_batch_kernels(const sffn_layer& L);
// Batched predictor (predict) and/or sparse FFN over the union (forward).
cudaError_t launch_batch(const sffn_layer& L, const float* x, int B, float thres, const sffn_masks* m, bool predict,
                         bool forward, float* y, float* x_out, void* ws, cudaStream_t st);

void set_error(const std::string& msg);
sffn_status cuda_fail(cudaError_t e, const char* what);

// Launchers (each enqueues kernels on `st`; they return the launch status).
cudaError_t launch_pred_hidden(const sffn_layer& L, const float* x, float* hid, cudaStream_t st);
cudaError_t launch_pred_scores(const sffn_layer& L, const float* hid, float thres, uint32_t* nmask,
                               cudaStream_t st);
cudaError_t launch_mask_views(const sffn_layer& L, const uint32_t* nmask, int32_t* idx, int32_t* count,
                              uint32_t* gmask, cudaStream_t st);
// `kept`: the workspace's per-block downT row counts (written and summed under zero-skip only).
cudaError_t launch_ffn(const sffn_layer& L, const float* x, const uint32_t* nmask, int32_t* idx_out,
                       int32_t* count_out, uint32_t* gmask_out, float* partials, int32_t* kept, cudaStream_t st);
cudaError_t launch_ffn_reduce(const sffn_layer& L, const float* partials, const int32_t* kept, const float* x,
                              float* y, float* x_out, cudaStream_t st);
cudaError_t launch_tam_update(tam_state& S, int layer0, int n_layers, const uint32_t* gmask, int gstride,
                              float lambda, float eps, int K, const tam_outputs& out, cudaStream_t st);
cudaError_t launch_tam_adapt(tam_state& S, int layer0, int n_layers, const uint8_t* stall, float alpha,
                             float lo, float hi, cudaStream_t st);
cudaError_t launch_selftest_timeout(uint32_t* err, int limit_us, cudaStream_t st);

// Whole-stack decode kernel (stack.cu).
constexpr size_t kStackBarBytes = 256;   // grid barrier words
bool stack_supported(const sffn_layer& L, std::string* why);
cudaError_t configure_stack_kernels(const sffn_layer& L);
size_t stack_ws_bytes(const sffn_layer& L);
size_t stack_layer_desc_bytes();
void stack_fill_layer_desc(const sffn_layer& L, void* out);
cudaError_t launch_stack(const sffn_stack& S, const float* x0, float* xs, float* ys, float thres,
                         const sffn_masks& m, void* ws, cudaStream_t st);

// Packing (setup).
// up_s, gate_s, down_s: per-neuron scales of SFFN_FFN_Q8 / Q4 rows (original order), else null.
sffn_status pack_layer(sffn_layer& L, const void* W1, const float* b1, const void* W2, const float* b2,
                       const void* up, const void* gate, const void* down, const int32_t* perm,
                       cudaStream_t st, const float* up_s = nullptr, const float* gate_s = nullptr,
                       const float* down_s = nullptr);

// Shared memory sizes, set as kernel attributes at layer creation.
cudaError_t configure_kernels(sffn_layer& L);
cudaError_t configure_predict_kernels(const sffn_layer& L);
int score_stages_for(const sffn_layer& L);
size_t score_smem(const sffn_layer& L);
int ffn_stages_for(const sffn_layer& L);
size_t ffn_smem(const sffn_layer& L);
int ffn_blocks(const sffn_layer& L);

// Records the layer's trace event for kernel slot k (if any) around `launch`.
template <typename F>
cudaError_t traced_batch(const sffn_layer& L, int k, cudaStream_t st, F&& launch) {
  cudaError_t e = cudaSuccess;
  if (L.trace_begin[k]) e = cudaEventRecord(L.trace_begin[k], st);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess && L.trace_end[k]) e = cudaEventRecord(L.trace_end[k], st);
  return e;
}

// Launch helper: programmatic dependent launch and optional cluster size.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      bool pdl, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster_x;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace sffn
