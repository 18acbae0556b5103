/*
 * sffn.h -- C ABI of libsffn.so: predictor-gated, activation-sparse FFN decode
 * on one GB300 (sm_103a), with group momentum (TAM) bookkeeping.
 *
 * Sources of the operations (page title, section):
 *   PowerInfer (SOSP'24) summary page -- §5.1 per-layer MLP predictor
 *     scores = W2 . ReLU(W1 . x); "Paper vs code": a neuron is computed iff
 *     score >= threshold (default 0.0); §5.2 neuron table mapping packed slots
 *     to the original matrix order; §5.3-§5.4 neuron-aware operators that
 *     touch only active rows (up/gate) and columns (down), each thread block on
 *     a disjoint neuron set; activation note: ReLU, ReGLU, SiLU-family.
 *   KAIROX (OSDI'26) review page -- 核心方法 item 1/3: co-activation groups
 *     stored as contiguous regions, at most 1024 groups per layer; item 4:
 *     temporal activation momentum (TAM), candidates above
 *     tau = (1 - lambda) + eps, highest scores kept within the budget;
 *     item 5: Adaptive Neuron Balancer (lambda up on I/O stall, down on compute
 *     stall); item 6: fused XOR/AND set update.
 *
 * Conventions for every call:
 *   - Device pointers are plain CUDA device addresses on the CURRENT device;
 *     host pointers are marked "host". Sizes are element counts unless named
 *     *_bytes. The caller owns every per-call buffer; handles own the packed
 *     weights and the momentum state.
 *   - Index space is packed-slot order: slot s holds original neuron perm[s].
 *     Neuron bitmask: slot i is bit (i % 32) of word (i / 32). Group bitmask:
 *     group g is bit (g % 32) of word (g / 32). Group g = slots
 *     [g*G, (g+1)*G). A group is active iff any of its slots is active.
 *   - Hot calls (sffn_predict, sffn_forward, sffn_decode_step, tam_update,
 *     tam_adapt) allocate nothing, never synchronize, only enqueue on the given
 *     stream, and may be captured in a CUDA graph. They use programmatic
 *     dependent launch between their own kernels.
 *   - Errors are returned as sffn_status, never raised: argument checks are
 *     synchronous and happen before any device work; a failed launch returns
 *     SFFN_ERR_CUDA; conditions found on the device (a bounded wait that ran
 *     out, an out-of-range index) set the handle's device error word, read by
 *     sffn_layer_check_error / tam_check_error. sffn_last_error() gives a
 *     thread-local description of the last failure.
 */
#ifndef SFFN_H_
#define SFFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sffn_stream;   /* == cudaStream_t; NULL = legacy default stream */

typedef enum {
  SFFN_OK = 0,
  SFFN_ERR_INVALID_ARG = 1,   /* a pointer, size, alignment or enum is not allowed */
  SFFN_ERR_UNSUPPORTED = 2,   /* valid, but not implemented by this build */
  SFFN_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  SFFN_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out */
  SFFN_ERR_OOM = 5,           /* device allocation failed (create/pack only) */
  SFFN_ERR_DEVICE = 6         /* the device found bad data (e.g. perm not a permutation) */
} sffn_status;

/* h = ReLU(u) | ReLU(g) * u | SiLU(g) * u | ReLU(u)^2 (squared ReLU, PowerInfer's
 * "Paper vs code" list), with u = up . x and g = gate . x; only ReGLU and
 * SwiGLU read gate rows. */
typedef enum { SFFN_ACT_RELU = 0, SFFN_ACT_REGLU = 1, SFFN_ACT_SWIGLU = 2, SFFN_ACT_RELU2 = 3 } sffn_act;
typedef enum { SFFN_F32 = 0, SFFN_F16 = 1, SFFN_BF16 = 2 } sffn_dtype;

/* Storage of the FFN rows (up, gate, down): in the layer's wdtype, or as 8-bit
 * or 4-bit codes with one fp32 scale per neuron (weight = code x scale; the
 * quantized models the pages run, e.g. PowerInfer's OPT-30B-Q4). SFFN_FFN_Q4
 * stores two signed 4-bit codes per byte, element 2i in the low half of byte
 * i. The predictor (W1, W2) always uses wdtype. */
typedef enum { SFFN_FFN_ROWS = 0, SFFN_FFN_Q8 = 1, SFFN_FFN_Q4 = 2 } sffn_ffn_format;

/* Shape of one FFN layer and its predictor.
 *   d: model dimension, multiple of 8, 8 <= d <= 16384.
 *   f: FFN neurons, multiple of group_size, f / group_size <= 1024 groups.
 *   h: predictor hidden size, multiple of 8, h * element size <= 2 KB
 *      (h <= 1024 for 16-bit weights, h <= 512 for fp32).
 *   group_size: 32 or 64 (KAIROX groups).
 *   act: sffn_act. ReLU and squared ReLU read up and down; ReGLU and SwiGLU also read gate.
 *   wdtype: storage type of every weight matrix (fp32 accumulation always).
 *   max_batch: largest B the layer will be called with, 1..32. */
typedef struct {
  int32_t d, f, h, group_size;
  int32_t act;
  int32_t wdtype;
  int32_t max_batch;
  int32_t ffn_format;   /* sffn_ffn_format; SFFN_FFN_Q8 needs wdtype fp16/bf16 and d % 16 == 0,
                           SFFN_FFN_Q4 fp16/bf16 and d % 32 == 0; batched calls (B > 1)
                           are not implemented for either */
} sffn_layer_desc;

/* One token's (or a batch's) active-set views, all device buffers owned by the
 * caller. Per-token arrays are laid out [B][...] with the stated row length:
 *   nmask  [B][f/32]      neuron bitmask
 *   gmask  [B][gw]        group bitmask, gw = ceil((f/G)/32)
 *   idx    [B][f]         ascending active slots; entries past count[b] are untouched
 *   count  [B]            number of active slots
 * Batch union (only read or written when B > 1; may be NULL when B == 1):
 *   unmask [f/32], ugmask [gw], uidx [f], ucount [1]. */
typedef struct {
  uint32_t* nmask;
  uint32_t* gmask;
  int32_t* idx;
  int32_t* count;
  uint32_t* unmask;
  uint32_t* ugmask;
  int32_t* uidx;
  int32_t* ucount;
} sffn_masks;

typedef struct sffn_layer sffn_layer;
typedef struct tam_state tam_state;

/* Device addresses of a layer's packed arrays (read-only view, for tests and
 * tools): W1 [h][d], b1 [h] (fp32, zeros if none), W2 [f][h] in slot order,
 * b2 [f] (fp32, slot order, zeros if none), up/gate/downT [f][d] in slot order
 * (gate NULL for ReLU and squared ReLU; downT[s][:] is column perm[s] of down), perm [f]. */
typedef struct {
  const void* W1;
  const float* b1;
  const void* W2;
  const float* b2;
  const void* up;
  const void* gate;
  const void* downT;
  const int32_t* perm;
  /* SFFN_FFN_Q8 / SFFN_FFN_Q4 only (NULL otherwise): per-slot scales of up, gate, downT rows */
  const float* up_scale;
  const float* gate_scale;
  const float* down_scale;
} sffn_packed_view;

/* ---------------------------------------------------------------- status */

const char* sffn_status_string(sffn_status s);
/* Thread-local text of the last failure in this thread ("" if none). */
const char* sffn_last_error(void);
/* Library version string, e.g. "sffn 0.1 sm_103a". */
const char* sffn_version(void);

/* ---------------------------------------------------------------- layers */

/* Host-only check of a layer description (no CUDA call). */
sffn_status sffn_layer_validate(const sffn_layer_desc* desc);

/* Create a layer on the current device: allocates the packed weight arrays
 * (uninitialised until sffn_layer_pack) and a device error word. *out is set
 * only on success. Errors: INVALID_ARG (desc), OOM, CUDA. */
sffn_status sffn_layer_create(const sffn_layer_desc* desc, sffn_layer** out);

/* Pack row-major weights into the grouped, neuron-major layout (setup, not a
 * hot call; synchronizes the stream before returning):
 *   W1 [h][d], W2 [f][h] (row n = original neuron n), up [f][d],
 *   gate [f][d] (NULL for ReLU and squared ReLU, required otherwise), down [d][f] (column n =
 *   original neuron n), all in the layer's wdtype; b1 [h], b2 [f] fp32 or NULL
 *   (zero); perm [f] int32 with perm[slot] = original neuron id, or NULL for
 *   the identity. Slot s of the packed arrays holds neuron perm[s]; down is
 *   stored transposed so each neuron's output column is one contiguous row.
 * Device pointers; 16-byte aligned. Errors: INVALID_ARG, DEVICE (perm is not
 * a permutation of 0..f-1), OOM (temporary buffer), CUDA. */
sffn_status sffn_layer_pack(sffn_layer* layer, const void* W1, const float* b1, const void* W2,
                            const float* b2, const void* up, const void* gate, const void* down,
                            const int32_t* perm, sffn_stream stream);

/* sffn_layer_pack for an SFFN_FFN_Q8 layer: W1, b1, W2, b2, perm as there;
 * up_q, gate_q [f][d] int8 codes with up_scale, gate_scale [f] fp32 (one per
 * neuron row), down_q [d][f] int8 codes with down_scale [f] fp32 (one per
 * neuron column), all in original neuron order; gate_q and gate_scale NULL
 * for ReLU and squared ReLU. Packed like sffn_layer_pack (slot order, down
 * transposed); the scales follow their rows. Device pointers, 16-byte
 * aligned. Errors: INVALID_ARG (also: the layer is not SFFN_FFN_Q8), DEVICE,
 * OOM, CUDA. The plain sffn_layer_pack rejects SFFN_FFN_Q8 layers. */
sffn_status sffn_layer_pack_q8(sffn_layer* layer, const void* W1, const float* b1, const void* W2,
                               const float* b2, const int8_t* up_q, const float* up_scale, const int8_t* gate_q,
                               const float* gate_scale, const int8_t* down_q, const float* down_scale,
                               const int32_t* perm, sffn_stream stream);

/* sffn_layer_pack_q8 for an SFFN_FFN_Q4 layer: the same arguments, with every
 * code in [-8, 7] (one int8 per code; the library packs two per byte). A code
 * outside that range fails with DEVICE and leaves the layer unpacked.
 * Errors: INVALID_ARG (also: the layer is not SFFN_FFN_Q4), DEVICE, OOM, CUDA. */
sffn_status sffn_layer_pack_q4(sffn_layer* layer, const void* W1, const float* b1, const void* W2,
                               const float* b2, const int8_t* up_q, const float* up_scale, const int8_t* gate_q,
                               const float* gate_scale, const int8_t* down_q, const float* down_scale,
                               const int32_t* perm, sffn_stream stream);

sffn_status sffn_layer_get_desc(const sffn_layer* layer, sffn_layer_desc* out /* host */);
sffn_status sffn_layer_packed(const sffn_layer* layer, sffn_packed_view* out /* host */);

/* Bytes of device workspace that the hot calls need for batch size B
 * (0 if the arguments are invalid). The workspace is caller-owned scratch,
 * 256-byte aligned, reused across calls; its contents need no initialisation. */
size_t sffn_workspace_bytes(const sffn_layer* layer, int32_t B);

/* Synchronize the stream, then read and clear the layer's device error word:
 * OK, TIMEOUT (a bounded wait ran out) or DEVICE (bad data seen on device). */
sffn_status sffn_layer_check_error(const sffn_layer* layer, sffn_stream stream);

void sffn_layer_destroy(sffn_layer* layer);

/* Optional per-kernel timing hooks. Kernel slots for B = 1: 0 predictor
 * hidden layer, 1 predictor scores + threshold, 2 sparse FFN (gather of active
 * up/gate rows, activation, and the active downT rows into per-block partial
 * sums), 3 reduction of the partial sums into y (and x + y). For B > 1 the
 * slots time the four tensor-core products: 0 hidden, 1 scores, 2 up/gate
 * over the union rows, 3 down over the union rows. When set, every later hot call on this layer records
 * begin[k] on its stream right before launching kernel k and end[k] right
 * after it (NULL entries are skipped). The handles are cudaEvent_t values owned
 * by the caller, which must keep them alive while tracing is on. Recording
 * between two kernels removes their launch overlap, so traced timings bound
 * each kernel alone. Pass NULL to turn tracing off. Host only; not
 * thread-safe against hot calls on the same layer from other threads. */
typedef struct {
  void* begin[4];
  void* end[4];
} sffn_trace;

sffn_status sffn_layer_set_trace(sffn_layer* layer, const sffn_trace* trace /* host, or NULL */);

/* Optional L2 hint for a layer stack at B = 1. `next` names the layer whose
 * hot call follows this layer's on the same stream (in a stack: layer l + 1,
 * and for the last layer layer 0 of the next token), or NULL to turn the hint
 * off. Each block of this layer's sparse-FFN kernel then asks L2 to fetch its
 * share of next's predictor hidden-layer weights (W1, PowerInfer §5.1) once
 * it has issued the copies of its own rows, so that those bytes move while
 * other blocks finish and while the reduction runs; the next predictor then
 * reads them from L2. Results are unchanged (the
 * prefetch only warms the cache). The library does not own `next`: the caller
 * keeps it alive while the hint is set, or unsets it first. `next` must live
 * on the same device; it may equal `layer`. Host only.
 * Errors: INVALID_ARG (layer NULL, or next on another device). */
sffn_status sffn_layer_set_next(sffn_layer* layer, const sffn_layer* next /* or NULL */);

/* Optional hot-group residency in L2 (the single-GPU analogue of PowerInfer's
 * hot/cold neuron split, §3-§4, with L2 in place of the GPU and HBM in place of
 * the CPU; KAIROX's momentum picks the hot groups, 核心方法 item 4). resident is
 * a device bitset of the layer's groups, [ceil(n_groups / 32)] uint32 (for
 * instance one layer's row of tam_outputs.resident from tam_update with a
 * capacity sized to the L2 share it may hold), or NULL to turn the hint off.
 * The B = 1 sparse-FFN kernel reads it at every launch (so tam_update may
 * rewrite it on the same stream between calls) and reads the up/gate/downT
 * rows of predicted-active neurons in those groups with the L2 evict-last
 * priority, all other rows with evict-first, so that hot rows tend to be
 * served from L2 on the next tokens. Results are unchanged (cache priorities
 * only). The caller keeps the buffer alive while it is set. Host only.
 * Errors: INVALID_ARG (layer NULL, resident not 4-byte aligned). */
sffn_status sffn_layer_set_l2_resident(sffn_layer* layer, const uint32_t* resident /* device, or NULL */);

/* Optional actual-activation zero-skip (PowerInfer §5.4: a neuron-aware
 * operator checks whether a neuron is active and computes only the active
 * ones, here applied to the activation itself). With enable != 0, the B = 1
 * sparse FFN (sffn_forward, sffn_decode_step) reads the transposed-down row of
 * a predicted-active neuron only if its activation h is non-zero (ReLU or a
 * ReGLU gate that clamps to 0 gives h = 0, and h * downT_i adds nothing to y).
 * The up (and gate) rows of every predicted-active neuron are still read: h is
 * known only after them. y is unchanged up to the sign of a zero sum;
 * idx / count / gmask still describe the predicted mask. rows_read: optional
 * device int32, or NULL; each B = 1 FFN call then writes the number of
 * transposed-down rows it read (stream-ordered with the call). Off by default;
 * calls with B > 1 ignore it. The caller keeps rows_read alive while it is
 * set. Host only. Errors: INVALID_ARG (layer NULL, rows_read not 4-byte
 * aligned). */
sffn_status sffn_layer_set_zero_skip(sffn_layer* layer, int32_t enable, int32_t* rows_read /* device, or NULL */);

/* Optional B = 1 grid sizes, for running one layer's predictor and another
 * layer's sparse FFN at the same time on two streams (one-layer-ahead
 * prediction: KAIROX observes that adjacent layers see near-identical inputs,
 * so layer l + 1's active set can be predicted from layer l's input while
 * layer l's FFN runs). The sparse-FFN kernel holds one large-shared-memory
 * block per SM and the predictor-scores kernel likewise, so they can only
 * overlap on disjoint SMs: ffn_blocks limits the FFN kernel and score_blocks
 * the scores kernel of this layer to that many blocks (0 = one per SM, the
 * default). The predictor's hidden-layer kernel needs no limit (it shares
 * SMs). Masks do not depend on the grid; y may differ by fp32 rounding,
 * because the FFN's per-block partial sums change with the block count.
 * Host only; the workspace size (sffn_workspace_bytes) never grows.
 * Errors: INVALID_ARG (layer NULL, a count outside [0, number of SMs], or
 * too few FFN blocks for the layer's shared-memory ring). */
sffn_status sffn_layer_set_grid(sffn_layer* layer, int32_t ffn_blocks, int32_t score_blocks);

/* Which arithmetic serves batched calls (B > 1) on this layer. The batch
 * reads each row of the union of its tokens' active sets once (KAIROX 问题与
 * 动机: a batch activates the union of its tokens' neurons; PowerInfer §3.2
 * on batches below 32):
 *   SFFN_BATCH_TENSOR      every product on the tensor cores (tcgen05.mma over
 *                          the union rows, activations as 16-bit hi/lo parts);
 *   SFFN_BATCH_CUDA_CORES  for 2 <= B <= 4: fp32 FFMA on the CUDA cores, the
 *                          B = 1 kernels' structure with every token's x in
 *                          registers (16-bit SFFN_FFN_ROWS weights, d <= 8192;
 *                          otherwise UNSUPPORTED); B > 4 takes the tensor cores;
 *   SFFN_BATCH_AUTO        the default: the CUDA cores for B = 2 where they
 *                          apply, the tensor cores otherwise (measured on
 *                          GB300: the CUDA-core arm is faster at B = 2 and
 *                          slower from B = 3 on).
 * Results agree within the parity tolerances either way; both arms write the
 * same views. Host only. Errors: INVALID_ARG (layer NULL, unknown path). */
typedef enum { SFFN_BATCH_AUTO = 0, SFFN_BATCH_TENSOR = 1, SFFN_BATCH_CUDA_CORES = 2 } sffn_batch_path;
sffn_status sffn_layer_set_batch_path(sffn_layer* layer, int32_t path);

/* The arm that serves a batched call of B tokens on this layer under its
 * current setting: SFFN_BATCH_TENSOR or SFFN_BATCH_CUDA_CORES, or -1 when no
 * arm does (B outside [2, max_batch], or a layer the batched paths do not
 * take: such a call returns UNSUPPORTED). Host only. */
int32_t sffn_layer_batch_arm(const sffn_layer* layer, int32_t B);

/* ---------------------------------------------------------------- hot calls */

/* Predictor (PowerInfer §5.1 and the threshold note): for each token b,
 *   hid = ReLU(W1 . x_b + b1), s = W2 . hid + b2, slot i active iff s_i >= thres
 * (NaN is inactive), written as masks->nmask/gmask/idx/count for row b; for
 * B > 1 also the union views. x: [B][d] fp32 device, 16-byte aligned.
 * ws: workspace of at least sffn_workspace_bytes(layer, B).
 * Errors: INVALID_ARG, UNSUPPORTED (B beyond what this build implements), CUDA. */
sffn_status sffn_predict(const sffn_layer* layer, const float* x, int32_t B, float thres,
                         const sffn_masks* masks, void* ws, size_t ws_bytes, sffn_stream stream);

/* Sparse FFN over the active set given by masks->nmask (rows [B][f/32]; any
 * caller-made mask is allowed): for each token b,
 *   y_b = sum_{slot i active for b} act(gate_i . x_b, up_i . x_b) * downT_i
 * with act = ReLU(u) | ReLU(g)*u | SiLU(g)*u, fp32 accumulation, fixed
 * summation order (run-to-run bit-identical). Only active rows are read
 * (PowerInfer §5.4). y: [B][d] fp32. x_out: NULL, or [B][d] fp32 that receives
 * x + y (the residual stream of a layer stack). Other mask fields are ignored.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
sffn_status sffn_forward(const sffn_layer* layer, const float* x, int32_t B, const sffn_masks* masks,
                         float* y, float* x_out, void* ws, size_t ws_bytes, sffn_stream stream);

/* sffn_predict followed by sffn_forward on the predicted masks, as one
 * pipelined sequence of kernels. All mask views are written. */
sffn_status sffn_decode_step(const sffn_layer* layer, const float* x, int32_t B, float thres,
                             const sffn_masks* masks, float* y, float* x_out, void* ws,
                             size_t ws_bytes, sffn_stream stream);

/* sffn_decode_step for callers that cannot allocate device memory: a decode
 * loop that must never stall on an allocation (one can synchronize the whole
 * GPU), a runtime that reaches this library only through its C ABI and has no
 * CUDA allocator, or a process whose memory pool refuses new allocations once
 * serving starts. Same arguments and results as sffn_decode_step at B = 1,
 * minus the workspace: scratch comes from one 16 MiB device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits. B > 1 returns UNSUPPORTED (the batched path's scratch is not held in
 * the array). The array is enough for any valid layer at B = 1 on a GPU with
 * up to about 240 SMs (the per-block partial sums take SMs x d x 4 bytes, at
 * most 10 MB on a 152-SM GB300, so no valid layer reaches the limit there); a
 * layer needing more returns INVALID_ARG. The call allocates nothing and
 * records no sffn_layer_set_trace events. Its first call on each device looks
 * up the array's device address (cudaGetSymbolAddress), so make that first
 * call before any stream capture. All calls on a device share the array:
 * calls that can overlap on the GPU race on it and must be ordered by the
 * caller; nothing in it needs clearing between calls. The pages describe no
 * counterpart of this call; it exists for callers of this library. */
sffn_status sffn_decode_step_static_ws(const sffn_layer* layer, const float* x, int32_t B, float thres,
                                       const sffn_masks* masks, float* y, float* x_out, sffn_stream stream);

/* ---------------------------------------------------------------- whole stack */

/* A stack of layers decoded one token at a time by ONE kernel launch: for
 * every layer in order, the predictor (PowerInfer §5.1), the threshold, the
 * sparse FFN over the predicted rows (§5.3-§5.4) and the residual
 * x_{l+1} = x_l + y_l -- the computation of sffn_decode_step at B = 1 with
 * x_out chaining the layers, with the same summation orders (hid, masks,
 * index lists, y and x_{l+1} are bit-identical to that chain on the same
 * inputs). One thread block per SM runs the whole token; grid-wide barriers
 * separate the phases, and each block streams the next phases' predictor
 * weights while the barriers and the other phases run. The layers must
 * share d, f, h, group_size, act and storage, use 16-bit weights in
 * SFFN_FFN_ROWS form, and keep at most 32 KB per neuron of up/gate rows
 * (d <= 8192 for ReGLU/SwiGLU, d <= 16384 for ReLU); other shapes return
 * UNSUPPORTED (use the per-layer calls). The stack keeps the layers' packed
 * arrays' addresses, not the layers: they must outlive it (re-packing a layer
 * in place is fine). Per-layer options (sffn_layer_set_next, _set_grid,
 * _set_l2_resident, _set_zero_skip) do not apply to the stack kernel.
 * Errors: INVALID_ARG (NULL, n_layers outside [1, 4096], layers that differ
 * or live on other devices), UNSUPPORTED, OOM, CUDA. */
typedef struct sffn_stack sffn_stack;
sffn_status sffn_stack_create(const sffn_layer* const* layers /* host array [n_layers] */, int32_t n_layers,
                              sffn_stack** out);

/* Bytes of caller workspace sffn_stack_decode needs (0 if stack is NULL):
 * the hidden vector and one partial sum of y per SM. */
size_t sffn_stack_workspace_bytes(const sffn_stack* stack);

/* One decode token through every layer (device pointers, fp32):
 *   x0  [d]            input of layer 0 (16-byte aligned); it may be one of
 *                      xs's rows, e.g. the previous token's output
 *                      xs + (n_layers-1)*d, and is otherwise not written;
 *   xs  [n_layers][d]  written: xs[l] = x_l + y_l, the input of layer l+1
 *                      (x_0 = x0); xs[n_layers-1] is the token's output;
 *   ys  [n_layers][d]  written if not NULL: y_l;
 *   masks: each field is a per-layer array, rows [n_layers][...] as for one
 *     token: nmask [n_layers][f/32] (required), gmask [n_layers][gw],
 *     idx [n_layers][f], count [n_layers] (each optional, NULL = not
 *     written); the union fields are ignored.
 *   ws: at least sffn_stack_workspace_bytes(stack), 256-byte aligned.
 * The kernel's grid barrier state lives in the stack handle, so calls on one
 * stack must not overlap on the GPU (order them on one stream); different
 * stacks may run concurrently only if the GPU can hold both grids, which one
 * GB300 cannot (each holds every SM). The launch needs every SM: work that
 * occupies SMs at the same time only delays it. Allocates nothing, does not
 * synchronize, may be captured in a CUDA graph. A bounded wait that runs out
 * is reported by sffn_stack_check_error.
 * Errors: INVALID_ARG, CUDA. */
sffn_status sffn_stack_decode(const sffn_stack* stack, const float* x0, float* xs, float* ys, float thres,
                              const sffn_masks* masks, void* ws, size_t ws_bytes, sffn_stream stream);

/* Synchronize the stream, read and clear the stack's device error word (OK,
 * TIMEOUT or DEVICE); after an error it also resets the grid barrier so the
 * next call starts clean. */
sffn_status sffn_stack_check_error(const sffn_stack* stack, sffn_stream stream);
void sffn_stack_destroy(sffn_stack* stack);

/* ---------------------------------------------------------------- TAM */

/* Momentum state for n_layers layers of n_groups groups (1..1024): scores
 * (fp32, start 0), lambda per layer (start lambda0, in (0, 1)), resident
 * bitset (start empty), and a device error word. */
sffn_status tam_create(int32_t n_layers, int32_t n_groups, float lambda0, tam_state** out);

/* Outputs of tam_update; every pointer is optional (NULL = not written).
 * Per-layer rows, n_layers rows each: bitsets [n][gw] with gw =
 * ceil(n_groups/32); topk [n][capacity_k] group ids in rank order (score
 * descending, then group id ascending), entries past n_res are -1;
 * n_cand [n], n_res [n]. */
typedef struct {
  uint32_t* cand;
  uint32_t* resident;
  uint32_t* load;
  uint32_t* evict;
  uint32_t* changed;
  int32_t* topk;
  int32_t* n_cand;
  int32_t* n_res;
} tam_outputs;

/* One momentum step for layers [layer0, layer0 + n_layers) (KAIROX 核心方法
 * item 4), float32 with one rounding per operation and no fused multiply-add:
 *   om = 1 - lambda; tau = om + eps;
 *   s_g = lambda * s_g;  s_g = s_g + (group g active ? om : 0);
 *   cand = {g : s_g > tau};  resident = the first capacity_k of cand ranked by
 *   (s_g descending, g ascending);  load = res & ~prev;  evict = prev & ~res;
 *   changed = res ^ prev;  the state's resident set becomes res.
 * gmask: device, row l (for layer layer0 + l) starts at gmask + l*gmask_stride
 * (words), gmask_stride >= gw. lambda < 0 uses each layer's state lambda.
 * eps >= 0, capacity_k in [0, n_groups]. One thread block per layer.
 * Errors: INVALID_ARG, CUDA. */
sffn_status tam_update(tam_state* tam, int32_t layer0, int32_t n_layers, const uint32_t* gmask,
                       int32_t gmask_stride, float lambda, float eps, int32_t capacity_k,
                       const tam_outputs* out, sffn_stream stream);

/* The whole per-layer decode step as the pages order it: the predictor, the
 * sparse FFN on the predicted masks (sffn_decode_step), then one momentum
 * step of layer `layer_index` of `tam` (tam_update with layer0 = layer_index,
 * n_layers = 1) on the group bitmask this call writes: masks->gmask for B = 1, the batch
 * union masks->ugmask for B > 1 (KAIROX 核心方法 item 4: the momentum of every
 * group is updated at every token from the predicted need; PowerInfer §5.1
 * for the predictor). All three are enqueued on `stream` in that order. The
 * momentum arguments mean what they mean for tam_update; `out` may be NULL.
 * The state must have the layer's group count and live on the same device.
 * Equivalent to sffn_decode_step followed by tam_update on the same stream;
 * a caller running many layers may instead batch the momentum steps of all
 * layers into one tam_update per token on a second stream (same results).
 * Errors: as sffn_decode_step and tam_update, and INVALID_ARG when the needed
 * group bitmask pointer is NULL. */
sffn_status sffn_decode_step_tam(const sffn_layer* layer, tam_state* tam, int32_t layer_index, const float* x,
                                 int32_t B, float thres, const sffn_masks* masks, float* y, float* x_out,
                                 void* ws, size_t ws_bytes, float lambda, float eps, int32_t capacity_k,
                                 const tam_outputs* out, sffn_stream stream);

/* Adaptive Neuron Balancer step (KAIROX 核心方法 item 5) for layers
 * [layer0, layer0 + n_layers): lambda_l <- min(hi, max(lo, lambda_l + (stall[l] ?
 * +alpha : -alpha))) in float32, where stall [n_layers] uint8 device (nonzero =
 * I/O stall). Requires 0 < lo <= hi < 1, alpha >= 0. */
sffn_status tam_adapt(tam_state* tam, int32_t layer0, int32_t n_layers, const uint8_t* stall,
                      float alpha, float lo, float hi, sffn_stream stream);

/* Copy the state out of / into caller device buffers (checkpoint / resume):
 * scores [n_layers][n_groups] fp32, lambdas [n_layers] fp32,
 * resident [n_layers][gw] u32. Any pointer may be NULL (skipped). */
sffn_status tam_get_state(const tam_state* tam, float* scores, float* lambdas, uint32_t* resident,
                          sffn_stream stream);
sffn_status tam_set_state(tam_state* tam, const float* scores, const float* lambdas,
                          const uint32_t* resident, sffn_stream stream);
sffn_status tam_get_shape(const tam_state* tam, int32_t* n_layers /* host */, int32_t* n_groups /* host */);
sffn_status tam_check_error(const tam_state* tam, sffn_stream stream);
void tam_destroy(tam_state* tam);

/* ---------------------------------------------------------------- self-test */

/* Exercise the bounded-wait path without any fault: one thread block waits
 * on a shared-memory barrier that nothing will complete, gives up after
 * limit_us microseconds (1..100000), records SFFN_ERR_TIMEOUT in the layer's
 * device error word and returns. sffn_layer_check_error then reports TIMEOUT
 * and the context stays usable. */
sffn_status sffn_selftest_wait_timeout(const sffn_layer* layer, int32_t limit_us, sffn_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* SFFN_H_ */
