"""ctypes binding of libsffn.so (include/sffn.h): argument marshalling only.

Every function named like a C entry point takes torch tensors (or None) where
the C call takes device pointers, passes ``tensor.data_ptr()`` and the current
torch CUDA stream, and raises :class:`SffnError` when the call returns a
status other than SFFN_OK. All arithmetic happens in the CUDA kernels behind
the C ABI; importing this module fails if the library has not been built.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libsffn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python -m activation_sparse_ffn_gb300.build`")

_lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- enums

SFFN_OK = 0
SFFN_ERR_INVALID_ARG = 1
SFFN_ERR_UNSUPPORTED = 2
SFFN_ERR_CUDA = 3
SFFN_ERR_TIMEOUT = 4
SFFN_ERR_OOM = 5
SFFN_ERR_DEVICE = 6

ACT = {"relu": 0, "reglu": 1, "swiglu": 2, "relu2": 3}
DTYPE = {"f32": 0, "f16": 1, "bf16": 2}
TORCH_WDTYPE = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}

# ----------------------------------------------------------------- structs

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class LayerDesc(ctypes.Structure):
    _fields_ = [("d", _i32), ("f", _i32), ("h", _i32), ("group_size", _i32), ("act", _i32), ("wdtype", _i32),
                ("max_batch", _i32), ("ffn_format", _i32)]


class MasksC(ctypes.Structure):
    _fields_ = [("nmask", _vp), ("gmask", _vp), ("idx", _vp), ("count", _vp), ("unmask", _vp), ("ugmask", _vp),
                ("uidx", _vp), ("ucount", _vp)]


class PackedView(ctypes.Structure):
    _fields_ = [("W1", _vp), ("b1", _vp), ("W2", _vp), ("b2", _vp), ("up", _vp), ("gate", _vp), ("downT", _vp),
                ("perm", _vp), ("up_scale", _vp), ("gate_scale", _vp), ("down_scale", _vp)]


class TraceC(ctypes.Structure):
    _fields_ = [("begin", _vp * 4), ("end", _vp * 4)]


class TamOutputsC(ctypes.Structure):
    _fields_ = [("cand", _vp), ("resident", _vp), ("load", _vp), ("evict", _vp), ("changed", _vp), ("topk", _vp),
                ("n_cand", _vp), ("n_res", _vp)]


def _sig(name, restype, *argtypes):
    fn = getattr(_lib, name)
    fn.restype = restype
    fn.argtypes = list(argtypes)
    return fn


_c = ctypes.c_int
_size = ctypes.c_size_t
_f32 = ctypes.c_float
_P = ctypes.POINTER

_sig("sffn_status_string", ctypes.c_char_p, _c)
_sig("sffn_last_error", ctypes.c_char_p)
_sig("sffn_version", ctypes.c_char_p)
_sig("sffn_layer_validate", _c, _P(LayerDesc))
_sig("sffn_layer_create", _c, _P(LayerDesc), _P(_vp))
_sig("sffn_layer_pack", _c, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("sffn_layer_get_desc", _c, _vp, _P(LayerDesc))
_sig("sffn_layer_packed", _c, _vp, _P(PackedView))
_sig("sffn_workspace_bytes", _size, _vp, _i32)
_sig("sffn_layer_set_trace", _c, _vp, _P(TraceC))
_sig("sffn_layer_set_next", _c, _vp, _vp)
_sig("sffn_layer_pack_q8", _c, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("sffn_layer_pack_q4", _c, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("sffn_layer_set_grid", _c, _vp, _i32, _i32)
_sig("sffn_layer_set_l2_resident", _c, _vp, _vp)
_sig("sffn_layer_set_zero_skip", _c, _vp, _i32, _vp)
_sig("sffn_layer_set_batch_path", _c, _vp, _i32)
_sig("sffn_layer_batch_arm", _i32, _vp, _i32)
_sig("sffn_layer_check_error", _c, _vp, _vp)
_sig("sffn_layer_destroy", None, _vp)
_sig("sffn_predict", _c, _vp, _vp, _i32, _f32, _P(MasksC), _vp, _size, _vp)
_sig("sffn_forward", _c, _vp, _vp, _i32, _P(MasksC), _vp, _vp, _vp, _size, _vp)
_sig("sffn_decode_step", _c, _vp, _vp, _i32, _f32, _P(MasksC), _vp, _vp, _vp, _size, _vp)
_sig("sffn_decode_step_static_ws", _c, _vp, _vp, _i32, _f32, _P(MasksC), _vp, _vp, _vp)
_sig("sffn_decode_step_tam", _c, _vp, _vp, _i32, _vp, _i32, _f32, _P(MasksC), _vp, _vp, _vp, _size, _f32, _f32, _i32,
     _P(TamOutputsC), _vp)
_sig("sffn_stack_create", _c, _P(_vp), _i32, _P(_vp))
_sig("sffn_stack_workspace_bytes", _size, _vp)
_sig("sffn_stack_decode", _c, _vp, _vp, _vp, _vp, _f32, _P(MasksC), _vp, _size, _vp)
_sig("sffn_stack_check_error", _c, _vp, _vp)
_sig("sffn_stack_destroy", None, _vp)
_sig("tam_create", _c, _i32, _i32, _f32, _P(_vp))
_sig("tam_update", _c, _vp, _i32, _i32, _vp, _i32, _f32, _f32, _i32, _P(TamOutputsC), _vp)
_sig("tam_adapt", _c, _vp, _i32, _i32, _vp, _f32, _f32, _f32, _vp)
_sig("tam_get_state", _c, _vp, _vp, _vp, _vp, _vp)
_sig("tam_set_state", _c, _vp, _vp, _vp, _vp, _vp)
_sig("tam_get_shape", _c, _vp, _P(_i32), _P(_i32))
_sig("tam_check_error", _c, _vp, _vp)
_sig("tam_destroy", None, _vp)
_sig("sffn_selftest_wait_timeout", _c, _vp, _i32, _vp)

EXPORTS = [
    "sffn_status_string", "sffn_last_error", "sffn_version", "sffn_layer_validate", "sffn_layer_create",
    "sffn_layer_pack", "sffn_layer_get_desc", "sffn_layer_packed", "sffn_workspace_bytes", "sffn_layer_set_trace", "sffn_layer_set_next", "sffn_layer_set_grid",
    "sffn_layer_set_l2_resident", "sffn_layer_set_zero_skip", "sffn_layer_set_batch_path", "sffn_layer_batch_arm",
    "sffn_layer_pack_q8", "sffn_layer_pack_q4",
    "sffn_layer_check_error",
    "sffn_layer_destroy", "sffn_predict", "sffn_forward", "sffn_decode_step", "sffn_decode_step_static_ws", "sffn_decode_step_tam",
    "sffn_stack_create", "sffn_stack_workspace_bytes", "sffn_stack_decode", "sffn_stack_check_error",
    "sffn_stack_destroy", "tam_create", "tam_update",
    "tam_adapt", "tam_get_state", "tam_set_state", "tam_get_shape", "tam_check_error", "tam_destroy",
    "sffn_selftest_wait_timeout",
]


class SffnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = _lib.sffn_status_string(status).decode()
        detail = _lib.sffn_last_error().decode()
        super().__init__(f"{where}: {self.name}: {detail}")


def _check(status: int, where: str) -> None:
    if status != SFFN_OK:
        raise SffnError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(status: int) -> str:
    return _lib.sffn_status_string(status).decode()


def last_error() -> str:
    return _lib.sffn_last_error().decode()


def version() -> str:
    return _lib.sffn_version().decode()


# ----------------------------------------------------------------- layer calls

FFN_FORMAT = {"rows": 0, "q8": 1, "q4": 2}


def make_desc(d, f, h, group_size, act, wdtype, max_batch=1, ffn_format="rows") -> LayerDesc:
    return LayerDesc(d, f, h, group_size, ACT[act] if isinstance(act, str) else act,
                     DTYPE[wdtype] if isinstance(wdtype, str) else wdtype, max_batch,
                     FFN_FORMAT[ffn_format] if isinstance(ffn_format, str) else ffn_format)


def sffn_layer_validate(desc: LayerDesc) -> int:
    """Host-only check; returns the status code (no exception)."""
    return _lib.sffn_layer_validate(ctypes.byref(desc))


def sffn_layer_create(desc: LayerDesc) -> int:
    h = _vp()
    _check(_lib.sffn_layer_create(ctypes.byref(desc), ctypes.byref(h)), "sffn_layer_create")
    return h.value


def sffn_layer_pack(layer, W1, b1, W2, b2, up, gate, down, perm, stream=None) -> None:
    _check(_lib.sffn_layer_pack(layer, _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(up), _ptr(gate), _ptr(down),
                                _ptr(perm), _stream(stream)), "sffn_layer_pack")


def sffn_layer_pack_q8(layer, W1, b1, W2, b2, up_q, up_s, gate_q, gate_s, down_q, down_s, perm, stream=None) -> None:
    _check(_lib.sffn_layer_pack_q8(layer, _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(up_q), _ptr(up_s), _ptr(gate_q),
                                   _ptr(gate_s), _ptr(down_q), _ptr(down_s), _ptr(perm), _stream(stream)),
           "sffn_layer_pack_q8")


def sffn_layer_pack_q4(layer, W1, b1, W2, b2, up_q, up_s, gate_q, gate_s, down_q, down_s, perm, stream=None) -> None:
    """As sffn_layer_pack_q8, with int8 codes in [-8, 7] (packed two per byte by the library)."""
    _check(_lib.sffn_layer_pack_q4(layer, _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(up_q), _ptr(up_s), _ptr(gate_q),
                                   _ptr(gate_s), _ptr(down_q), _ptr(down_s), _ptr(perm), _stream(stream)),
           "sffn_layer_pack_q4")


def sffn_layer_get_desc(layer) -> LayerDesc:
    out = LayerDesc()
    _check(_lib.sffn_layer_get_desc(layer, ctypes.byref(out)), "sffn_layer_get_desc")
    return out


def sffn_layer_packed(layer) -> PackedView:
    out = PackedView()
    _check(_lib.sffn_layer_packed(layer, ctypes.byref(out)), "sffn_layer_packed")
    return out


TRACE_KERNELS = ("pred_hidden", "pred_scores", "ffn", "ffn_reduce")


def sffn_layer_set_trace(layer, begin=None, end=None) -> None:
    """begin/end: sequences of 4 torch.cuda.Event (or None) for the kernel
    slots in TRACE_KERNELS; both None turns tracing off. Each event is
    recorded once here first so that its CUDA handle exists."""
    if begin is None and end is None:
        _check(_lib.sffn_layer_set_trace(layer, None), "sffn_layer_set_trace")
        return
    t = TraceC()
    for k in range(4):
        for arr, evs in ((t.begin, begin), (t.end, end)):
            ev = evs[k] if evs is not None else None
            if ev is not None:
                ev.record()
                arr[k] = ev.cuda_event
    _check(_lib.sffn_layer_set_trace(layer, ctypes.byref(t)), "sffn_layer_set_trace")


def sffn_layer_set_next(layer, next_layer=None) -> None:
    """L2 hint: ``next_layer`` (a handle, or None) follows ``layer`` on the stream."""
    _check(_lib.sffn_layer_set_next(layer, next_layer), "sffn_layer_set_next")


def sffn_layer_set_grid(layer, ffn_blocks: int = 0, score_blocks: int = 0) -> None:
    """B = 1 grid sizes (0 = one block per SM), for predictor/FFN overlap."""
    _check(_lib.sffn_layer_set_grid(layer, ffn_blocks, score_blocks), "sffn_layer_set_grid")


def sffn_layer_set_l2_resident(layer, resident=None) -> None:
    """Hot-group bitset (device uint32 [ceil(n_groups/32)], or None) whose rows stay in L2."""
    _check(_lib.sffn_layer_set_l2_resident(layer, _ptr(resident)), "sffn_layer_set_l2_resident")


def sffn_layer_set_zero_skip(layer, enable: bool, rows_read=None) -> None:
    """Zero-skip of the B = 1 FFN (downT rows of neurons with h != 0 only); rows_read: device int32 or None."""
    _check(_lib.sffn_layer_set_zero_skip(layer, 1 if enable else 0, _ptr(rows_read)), "sffn_layer_set_zero_skip")


BATCH_PATH = {"auto": 0, "tensor": 1, "cuda_cores": 2}


def sffn_layer_set_batch_path(layer, path) -> None:
    """Arithmetic of batched calls: "auto", "tensor" or "cuda_cores" (2 <= B <= 4)."""
    _check(_lib.sffn_layer_set_batch_path(layer, BATCH_PATH[path] if isinstance(path, str) else path),
           "sffn_layer_set_batch_path")


def sffn_layer_batch_arm(layer, B: int) -> str | None:
    """"tensor" or "cuda_cores": the arm serving a batch of B on this layer now (None: no arm)."""
    a = int(_lib.sffn_layer_batch_arm(layer, B))
    return {1: "tensor", 2: "cuda_cores"}.get(a)


def sffn_workspace_bytes(layer, B: int) -> int:
    return int(_lib.sffn_workspace_bytes(layer, B))


def sffn_layer_check_error(layer, stream=None) -> None:
    _check(_lib.sffn_layer_check_error(layer, _stream(stream)), "sffn_layer_check_error")


def sffn_layer_destroy(layer) -> None:
    _lib.sffn_layer_destroy(layer)


def sffn_predict(layer, x, B, thres, masks: "Masks", ws, stream=None) -> None:
    _check(_lib.sffn_predict(layer, _ptr(x), B, thres, ctypes.byref(masks.c), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "sffn_predict")


def sffn_forward(layer, x, B, masks: "Masks", y, x_out, ws, stream=None) -> None:
    _check(_lib.sffn_forward(layer, _ptr(x), B, ctypes.byref(masks.c), _ptr(y), _ptr(x_out), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "sffn_forward")


def sffn_decode_step(layer, x, B, thres, masks: "Masks", y, x_out, ws, stream=None) -> None:
    _check(_lib.sffn_decode_step(layer, _ptr(x), B, thres, ctypes.byref(masks.c), _ptr(y), _ptr(x_out), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)), "sffn_decode_step")


def sffn_decode_step_static_ws(layer, x, B, thres, masks: "Masks", y, x_out, stream=None) -> None:
    """sffn_decode_step without a workspace argument: the scratch lives in a
    16 MiB device array inside the library, for callers that cannot allocate
    device memory. Calls sharing a device must not overlap on the GPU."""
    _check(_lib.sffn_decode_step_static_ws(layer, _ptr(x), B, thres, ctypes.byref(masks.c), _ptr(y), _ptr(x_out),
                                           _stream(stream)), "sffn_decode_step_static_ws")


def sffn_decode_step_tam(layer, tam, layer_index, x, B, thres, masks: "Masks", y, x_out, ws, lam, eps, capacity_k,
                         outputs: "TamOutputs | None", stream=None) -> None:
    """sffn_decode_step, then the momentum step of layer ``layer_index`` on the group bitmask it wrote."""
    oc = outputs.c if outputs is not None else TamOutputsC()
    _check(_lib.sffn_decode_step_tam(layer, tam, layer_index, _ptr(x), B, thres, ctypes.byref(masks.c), _ptr(y),
                                     _ptr(x_out), _ptr(ws), ws.numel() * ws.element_size(), lam, eps, capacity_k,
                                     ctypes.byref(oc), _stream(stream)), "sffn_decode_step_tam")


def sffn_selftest_wait_timeout(layer, limit_us: int, stream=None) -> None:
    _check(_lib.sffn_selftest_wait_timeout(layer, limit_us, _stream(stream)), "sffn_selftest_wait_timeout")


# ----------------------------------------------------------------- whole-stack calls

def sffn_stack_create(layers) -> int:
    """layers: sequence of layer handles (ints)."""
    arr = (_vp * len(layers))(*layers)
    h = _vp()
    _check(_lib.sffn_stack_create(arr, len(layers), ctypes.byref(h)), "sffn_stack_create")
    return h.value


def sffn_stack_workspace_bytes(stack) -> int:
    return int(_lib.sffn_stack_workspace_bytes(stack))


def sffn_stack_decode(stack, x0, xs, ys, thres, masks: "StackMasks", ws, stream=None) -> None:
    _check(_lib.sffn_stack_decode(stack, _ptr(x0), _ptr(xs), _ptr(ys), thres, ctypes.byref(masks.c), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)), "sffn_stack_decode")


def sffn_stack_check_error(stack, stream=None) -> None:
    _check(_lib.sffn_stack_check_error(stack, _stream(stream)), "sffn_stack_check_error")


def sffn_stack_destroy(stack) -> None:
    _lib.sffn_stack_destroy(stack)


# ----------------------------------------------------------------- TAM calls

def tam_create(n_layers: int, n_groups: int, lambda0: float) -> int:
    h = _vp()
    _check(_lib.tam_create(n_layers, n_groups, lambda0, ctypes.byref(h)), "tam_create")
    return h.value


def tam_update(tam, layer0, n_layers, gmask, gmask_stride, lam, eps, capacity_k, outputs: "TamOutputs | None",
               stream=None) -> None:
    oc = outputs.c if outputs is not None else TamOutputsC()
    _check(_lib.tam_update(tam, layer0, n_layers, _ptr(gmask), gmask_stride, lam, eps, capacity_k, ctypes.byref(oc),
                           _stream(stream)), "tam_update")


def tam_adapt(tam, layer0, n_layers, stall, alpha, lo, hi, stream=None) -> None:
    _check(_lib.tam_adapt(tam, layer0, n_layers, _ptr(stall), alpha, lo, hi, _stream(stream)), "tam_adapt")


def tam_get_state(tam, scores, lambdas, resident, stream=None) -> None:
    _check(_lib.tam_get_state(tam, _ptr(scores), _ptr(lambdas), _ptr(resident), _stream(stream)), "tam_get_state")


def tam_set_state(tam, scores, lambdas, resident, stream=None) -> None:
    _check(_lib.tam_set_state(tam, _ptr(scores), _ptr(lambdas), _ptr(resident), _stream(stream)), "tam_set_state")


def tam_get_shape(tam) -> tuple[int, int]:
    a, b = _i32(), _i32()
    _check(_lib.tam_get_shape(tam, ctypes.byref(a), ctypes.byref(b)), "tam_get_shape")
    return a.value, b.value


def tam_check_error(tam, stream=None) -> None:
    _check(_lib.tam_check_error(tam, _stream(stream)), "tam_check_error")


def tam_destroy(tam) -> None:
    _lib.tam_destroy(tam)


# ----------------------------------------------------------------- buffers

class Masks:
    """Caller-owned mask buffers (torch int32 tensors on the device) and the
    C struct that points at them. Shapes follow include/sffn.h."""

    def __init__(self, f: int, group_size: int, B: int = 1, device="cuda"):
        n_groups = f // group_size
        self.f, self.group_size, self.B = f, group_size, B
        self.nwords, self.gwords = f // 32, (n_groups + 31) // 32
        kw = dict(dtype=torch.int32, device=device)
        self.nmask = torch.zeros(B, self.nwords, **kw)
        self.gmask = torch.zeros(B, self.gwords, **kw)
        self.idx = torch.full((B, f), -1, **kw)
        self.count = torch.zeros(B, **kw)
        self.unmask = torch.zeros(self.nwords, **kw)
        self.ugmask = torch.zeros(self.gwords, **kw)
        self.uidx = torch.full((f,), -1, **kw)
        self.ucount = torch.zeros(1, **kw)
        self.c = MasksC(*(t.data_ptr() for t in (self.nmask, self.gmask, self.idx, self.count, self.unmask,
                                                   self.ugmask, self.uidx, self.ucount)))


class StackMasks:
    """Per-layer mask buffers of sffn_stack_decode: nmask [L][f/32], gmask
    [L][gw], idx [L][f], count [L] (torch int32 on the device)."""

    def __init__(self, n_layers: int, f: int, group_size: int, device="cuda"):
        n_groups = f // group_size
        self.nwords, self.gwords = f // 32, (n_groups + 31) // 32
        kw = dict(dtype=torch.int32, device=device)
        self.nmask = torch.zeros(n_layers, self.nwords, **kw)
        self.gmask = torch.zeros(n_layers, self.gwords, **kw)
        self.idx = torch.full((n_layers, f), -1, **kw)
        self.count = torch.zeros(n_layers, **kw)
        self.c = MasksC(self.nmask.data_ptr(), self.gmask.data_ptr(), self.idx.data_ptr(), self.count.data_ptr(),
                        None, None, None, None)


class Stack:
    """Owns one sffn_stack handle over ``layers`` (Layer objects, kept alive)."""

    def __init__(self, layers):
        self.layers = list(layers)
        self.handle = sffn_stack_create([L.handle for L in self.layers])
        self.n_layers = len(self.layers)
        L0 = self.layers[0]
        self.d, self.f, self.group_size = L0.d, L0.f, L0.group_size

    def workspace(self, device="cuda") -> torch.Tensor:
        return torch.empty(sffn_stack_workspace_bytes(self.handle), dtype=torch.uint8, device=device)

    def masks(self, device="cuda") -> StackMasks:
        return StackMasks(self.n_layers, self.f, self.group_size, device)

    def check_error(self, stream=None) -> None:
        sffn_stack_check_error(self.handle, stream)

    def close(self) -> None:
        if getattr(self, "handle", None):
            sffn_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class TamOutputs:
    """Caller-owned output buffers of tam_update for n_layers layers."""

    def __init__(self, n_layers: int, n_groups: int, capacity_k: int, device="cuda"):
        gw = (n_groups + 31) // 32
        kw = dict(dtype=torch.int32, device=device)
        self.cand = torch.zeros(n_layers, gw, **kw)
        self.resident = torch.zeros(n_layers, gw, **kw)
        self.load = torch.zeros(n_layers, gw, **kw)
        self.evict = torch.zeros(n_layers, gw, **kw)
        self.changed = torch.zeros(n_layers, gw, **kw)
        self.topk = torch.full((n_layers, max(1, capacity_k)), -1, **kw)
        self.n_cand = torch.zeros(n_layers, **kw)
        self.n_res = torch.zeros(n_layers, **kw)
        self.c = TamOutputsC(*(t.data_ptr() for t in (self.cand, self.resident, self.load, self.evict, self.changed,
                                                        self.topk, self.n_cand, self.n_res)))


class Layer:
    """Owns one sffn_layer handle. ``weights`` holds device tensors in the
    original neuron order: W1 (h, d), W2 (f, h), up (f, d), gate (f, d) or
    None, down (d, f), perm (f,) int32, b1/b2 float32 or None; or, for 8-bit
    FFN rows, up_q/gate_q (f, d) and down_q (d, f) int8 with up_s/gate_s/down_s
    (f,) float32 scales in place of up/gate/down."""

    def __init__(self, d, f, h, group_size, act, wdtype, max_batch=1, ffn_format="rows"):
        self.desc = make_desc(d, f, h, group_size, act, wdtype, max_batch, ffn_format)
        self.ffn_format = ffn_format
        self.handle = sffn_layer_create(self.desc)
        self.d, self.f, self.h, self.group_size = d, f, h, group_size
        self.act, self.wdtype, self.max_batch = act, wdtype, max_batch

    @classmethod
    def from_weights(cls, weights: dict, group_size: int, act: str, max_batch=1, stream=None) -> "Layer":
        W1 = weights["W1"]
        q8 = weights.get("up_q") is not None
        up = weights["up_q"] if q8 else weights["up"]
        h, d = W1.shape
        f = up.shape[0]
        fmt = ("q4" if weights.get("qbits") == 4 else "q8") if q8 else "rows"
        layer = cls(d, f, h, group_size, act, TORCH_WDTYPE[W1.dtype], max_batch, fmt)
        layer.pack(weights, stream)
        return layer

    def pack(self, w: dict, stream=None) -> None:
        def c(t):
            return None if t is None else t.contiguous()
        perm = w.get("perm")
        perm = None if perm is None else c(perm.to(torch.int32))
        if w.get("up_q") is not None:
            pack = sffn_layer_pack_q4 if w.get("qbits") == 4 else sffn_layer_pack_q8
            pack(self.handle, c(w["W1"]), c(w.get("b1")), c(w["W2"]), c(w.get("b2")), c(w["up_q"]), c(w["up_s"]),
                 c(w.get("gate_q")), c(w.get("gate_s")), c(w["down_q"]), c(w["down_s"]), perm, stream)
        else:
            sffn_layer_pack(self.handle, c(w["W1"]), c(w.get("b1")), c(w["W2"]), c(w.get("b2")), c(w["up"]),
                            c(w.get("gate")), c(w["down"]), perm, stream)

    def workspace(self, B=1, device="cuda") -> torch.Tensor:
        n = sffn_workspace_bytes(self.handle, B)
        return torch.empty(n, dtype=torch.uint8, device=device)

    def masks(self, B=1, device="cuda") -> Masks:
        return Masks(self.f, self.group_size, B, device)

    def packed(self) -> PackedView:
        return sffn_layer_packed(self.handle)

    def check_error(self, stream=None) -> None:
        sffn_layer_check_error(self.handle, stream)

    def set_grid(self, ffn_blocks: int = 0, score_blocks: int = 0) -> None:
        sffn_layer_set_grid(self.handle, ffn_blocks, score_blocks)

    def set_l2_resident(self, resident) -> None:
        """Hot-group bitset (device tensor or pointer) of sffn_layer_set_l2_resident; keeps a tensor alive."""
        sffn_layer_set_l2_resident(self.handle, resident)
        self._resident = resident

    def set_zero_skip(self, enable: bool, rows_read=None) -> None:
        """sffn_layer_set_zero_skip; keeps a rows_read tensor alive while set."""
        sffn_layer_set_zero_skip(self.handle, enable, rows_read)
        self._rows_read = rows_read if enable else None

    def set_batch_path(self, path) -> None:
        sffn_layer_set_batch_path(self.handle, path)

    def set_next(self, other: "Layer | None") -> None:
        """L2 hint of sffn_layer_set_next; keeps ``other`` alive while set."""
        sffn_layer_set_next(self.handle, other.handle if other is not None else None)
        self._next = other

    def close(self) -> None:
        if getattr(self, "handle", None):
            sffn_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Tam:
    """Owns one tam_state handle."""

    def __init__(self, n_layers: int, n_groups: int, lambda0: float):
        self.handle = tam_create(n_layers, n_groups, lambda0)
        self.n_layers, self.n_groups = n_layers, n_groups

    def close(self) -> None:
        if getattr(self, "handle", None):
            tam_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DeviceArray:
    """Minimal __cuda_array_interface__ holder used to view a device address."""

    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 2, "strides": None}


_TYPESTR = {torch.float32: ("<f4", None), torch.float16: ("<f2", None), torch.int32: ("<i4", None),
            torch.bfloat16: ("<i2", torch.bfloat16), torch.uint8: ("|u1", None)}


def view_device(ptr: int, shape: tuple, dtype: torch.dtype) -> torch.Tensor:
    """A torch tensor aliasing device memory at ``ptr`` (no copy), e.g. one
    of the arrays of :func:`sffn_layer_packed`. The memory stays owned by the
    library handle; do not use the view after the handle is destroyed."""
    typestr, view_as = _TYPESTR[dtype]
    t = torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")
    return t.view(view_as) if view_as is not None else t
