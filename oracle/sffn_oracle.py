"""Plain CPU oracle of the predictor-gated, activation-sparse FFN decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import
this module. The product path (``activation_sparse_ffn_gb300``) never imports
it, and this module imports nothing from the product path: the two share no
code. Inputs come from the seeded generator or from the tests themselves.

Every function is a direct restatement of one step of the method, in float64
unless the step is an integer decision taken in float32 on purpose (the
temporal-activation-momentum update). No blocking, fusion or reordering beyond
what the definition states; numpy's matmul is used as a library primitive.

Sources (page title, then section):
  * PowerInfer (SOSP'24) summary page -- §5.1 "Predictors" (per-layer MLP
    predictor, scores = W2 . ReLU(W1 . x)), the "Paper vs code" note on the
    predictor threshold (a neuron is computed when score >= threshold, default
    0.0), §5.2 (neuron table mapping slots back to the original matrix order),
    §5.3/§5.4 (each side touches only the active rows of up/gate and the active
    columns of down; the hybrid merge sums the partials), §8.4 and the
    activation-function note (ReLU, ReGLU; SiLU-family models).
  * KAIROX (OSDI'26) review page -- 核心方法 items 1 and 3 (co-activation
    groups stored contiguously, at most 1024 groups per layer, GPU argsort and
    set difference), item 4 (temporal activation momentum, TAM: a group's
    score accumulates when active and decays by lambda when not; candidates are
    groups whose score exceeds tau = (1 - lambda) + eps; the highest-scoring
    candidates that fit the budget are kept; tau sits just above the score of
    one isolated activation), item 5 (Adaptive Neuron Balancer: an I/O stall
    raises lambda, a compute stall lowers it), item 6 (fused XOR/AND update).

Readings where the pages are silent are listed in the design notes; the ones
that change arithmetic are repeated at the function that applies them.
"""

from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# Stored weights
# --------------------------------------------------------------------------

DTYPES = ("f32", "f16", "bf16")


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Return the stored values of ``a`` exactly, as float64.

    ``dtype`` names how ``a`` is stored: ``"f32"`` (float32 array), ``"f16"``
    (float16 array) or ``"bf16"`` (uint16 array of bfloat16 bit patterns; a
    bfloat16 is the upper half of a float32, so shifting its bits left by 16
    gives that float32 exactly). Widening is exact for all three.
    """
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(a, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# Predictor (PowerInfer §5.1) and threshold
# --------------------------------------------------------------------------

def predictor_hidden(W1: np.ndarray, x: np.ndarray, b1: np.ndarray | None = None) -> np.ndarray:
    """Hidden layer of the per-layer MLP predictor: ReLU(W1 . x + b1).

    W1 is (h, d) float64, x is (d,) float64, b1 is (h,) or None (no bias, as
    in the page's pseudocode). Returns (h,) float64. PowerInfer §5.1.
    """
    pre = W1 @ x
    if b1 is not None:
        pre = pre + b1
    return np.maximum(pre, 0.0)


def predictor_scores(W2: np.ndarray, hid: np.ndarray, b2: np.ndarray | None = None) -> np.ndarray:
    """Output layer of the predictor: one score per FFN neuron, W2 . hid + b2.

    W2 is (n, h) float64 with one row per neuron, in whatever neuron order the
    caller uses; hid is (h,). PowerInfer §5.1.
    """
    s = W2 @ hid
    if b2 is not None:
        s = s + b2
    return s


def active_from_scores(scores: np.ndarray, thres: float) -> np.ndarray:
    """A neuron is computed iff its score is >= thres (PowerInfer, "Paper vs
    code": the released engine skips a neuron whose score is below the
    threshold, default 0.0). A NaN score compares false, so it is inactive."""
    with np.errstate(invalid="ignore"):
        return np.asarray(scores >= thres, dtype=bool)


# --------------------------------------------------------------------------
# Mask views: neuron bitmask, group bitmask, ascending index list
# --------------------------------------------------------------------------

def bits_to_words(bits: np.ndarray) -> np.ndarray:
    """Pack a bool vector into uint32 words: element i is bit (i % 32) of
    word (i // 32). The length must be a multiple of 32 after zero padding."""
    n = bits.shape[0]
    nw = (n + 31) // 32
    words = np.zeros(nw, dtype=np.uint32)
    for i in np.flatnonzero(bits):
        words[i // 32] |= np.uint32(1) << np.uint32(i % 32)
    return words


def words_to_bits(words: np.ndarray, n: int) -> np.ndarray:
    """Inverse of :func:`bits_to_words` for the first ``n`` elements."""
    out = np.zeros(n, dtype=bool)
    for i in range(n):
        out[i] = bool((int(words[i // 32]) >> (i % 32)) & 1)
    return out


def group_active(active: np.ndarray, group_size: int) -> np.ndarray:
    """A co-activation group (group_size contiguous slots, KAIROX 核心方法
    item 3) is active iff at least one of its neurons is active."""
    f = active.shape[0]
    if f % group_size:
        raise ValueError("f must be a multiple of the group size")
    return active.reshape(f // group_size, group_size).any(axis=1)


def mask_views(active: np.ndarray, group_size: int) -> dict:
    """All views of one token's active set, in packed-slot order.

    Returns nmask (uint32 words, f/32), gmask (uint32 words, ceil(n_groups/32)),
    idx (int32, ascending active slots) and count. Index-list order is
    ascending slot order (a reading: the pages leave it open).
    """
    g = group_active(active, group_size)
    idx = np.flatnonzero(active).astype(np.int32)
    return {
        "nmask": bits_to_words(active),
        "gmask": bits_to_words(g),
        "idx": idx,
        "count": int(idx.shape[0]),
    }


# --------------------------------------------------------------------------
# Sparse FFN over the active neurons (PowerInfer §5.3-§5.4)
# --------------------------------------------------------------------------

ACTS = ("relu", "reglu", "swiglu", "relu2")
GATED = ("reglu", "swiglu")   # activations that read a gate row


def activation(act: str, u: np.ndarray, g: np.ndarray | None) -> np.ndarray:
    """Per-neuron activation value h_i from the up value u_i and gate value g_i.

    relu:   h = max(0, u)                      (ReLU FFN, no gate)
    reglu:  h = max(0, g) * u                  (ReGLU)
    swiglu: h = g / (1 + exp(-g)) * u          (SiLU-gated, SwiGLU)
    relu2:  h = max(0, u)^2                    (squared ReLU, no gate)
    PowerInfer names the ReLU family and SiLU-based models (activation note,
    §4, §8.4); its "Paper vs code" list names ReLU, ReGLU and squared ReLU.
    """
    if act == "relu":
        return np.maximum(u, 0.0)
    if act == "relu2":
        r = np.maximum(u, 0.0)
        return r * r
    if act == "reglu":
        return np.maximum(g, 0.0) * u
    if act == "swiglu":
        return g / (1.0 + np.exp(-g)) * u
    raise ValueError(f"unknown activation {act!r}")


def ffn_sparse(x: np.ndarray, up: np.ndarray, gate: np.ndarray | None, down: np.ndarray,
               act: str, active: np.ndarray, perm: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray]:
    """y = sum over active neurons i of h_i * down[:, orig(i)].

    x (d,) float64. up, gate: (f, d) float64 in ORIGINAL neuron order (gate is
    None for ReLU). down: (d, f) float64 in original order (down[:, n] is
    neuron n's output column). active: (f,) bool in packed-SLOT order. perm:
    (f,) int, perm[slot] = original neuron id (the neuron table of PowerInfer
    §5.2); None means the identity.

    Only the active neurons' rows of up/gate and columns of down are read
    (PowerInfer §5.4). Returns (y (d,), h (n_active,) in ascending slot order).
    """
    f = up.shape[0]
    if perm is None:
        perm = np.arange(f)
    slots = np.flatnonzero(active)
    orig = np.asarray(perm)[slots]
    u = up[orig] @ x
    g = gate[orig] @ x if gate is not None else None
    h = activation(act, u, g)
    y = down[:, orig] @ h
    return y, h


def ffn_sparse_zero_skip(x: np.ndarray, up: np.ndarray, gate: np.ndarray | None, down: np.ndarray,
                         act: str, active: np.ndarray, perm: np.ndarray | None = None) -> tuple[np.ndarray, int]:
    """Zero-skip form of :func:`ffn_sparse`: the neuron-aware operator computes
    only the neurons that matter (PowerInfer §5.4), taken one step further to
    the activation itself. h is computed for every predicted-active neuron
    (its up and gate rows are read), then only the down columns of neurons
    with h_i != 0 are read (a NaN h is kept: it is not zero). Same arguments as
    ffn_sparse. Returns (y (d,), number of down columns read)."""
    f = up.shape[0]
    if perm is None:
        perm = np.arange(f)
    orig = np.asarray(perm)[np.flatnonzero(active)]
    u = up[orig] @ x
    g = gate[orig] @ x if gate is not None else None
    h = activation(act, u, g)
    keep = h != 0.0
    y = down[:, orig[keep]] @ h[keep]
    return y, int(keep.sum())


def ffn_sparse_stored(x: np.ndarray, up_s, gate_s, down_s, dtype: str, act: str, active: np.ndarray,
                      perm=None) -> tuple[np.ndarray, np.ndarray]:
    """:func:`ffn_sparse` on STORED weights (see :func:`widen`), widening only
    the active rows of up/gate and columns of down, which keeps full-size
    layers affordable. Same definition: the gathered rows are passed to
    ffn_sparse with every gathered neuron active."""
    f = up_s.shape[0]
    perm = np.arange(f) if perm is None else np.asarray(perm)
    orig = perm[np.flatnonzero(active)]
    U = widen(up_s[orig], dtype)
    G = widen(gate_s[orig], dtype) if gate_s is not None else None
    D = widen(down_s[:, orig], dtype)
    return ffn_sparse(x, U, G, D, act, np.ones(orig.shape[0], dtype=bool), None)


def ffn_sparse_q8(x: np.ndarray, up_q, up_scale, gate_q, gate_scale, down_q, down_scale, act: str,
                  active: np.ndarray, perm=None) -> tuple[np.ndarray, np.ndarray]:
    """:func:`ffn_sparse` on 8-bit quantized rows (the quantized models of the
    pages' Q4/Q8 runs, here one int8 code per weight and one float32 scale per
    neuron): the weight is code x scale. up_q, gate_q (f, d) int8 with
    up_scale, gate_scale (f,) float32, one per neuron row; down_q (d, f) int8
    with down_scale (f,) float32, one per neuron column; original neuron order.
    Only the active neurons' codes are widened (exactly, to float64)."""
    f = up_q.shape[0]
    perm = np.arange(f) if perm is None else np.asarray(perm)
    orig = perm[np.flatnonzero(active)]
    U = up_q[orig].astype(np.float64) * up_scale[orig].astype(np.float64)[:, None]
    G = None
    if gate_q is not None:
        G = gate_q[orig].astype(np.float64) * gate_scale[orig].astype(np.float64)[:, None]
    D = down_q[:, orig].astype(np.float64) * down_scale[orig].astype(np.float64)[None, :]
    return ffn_sparse(x, U, G, D, act, np.ones(orig.shape[0], dtype=bool), None)


def ffn_sparse_q4(x: np.ndarray, up_q, up_scale, gate_q, gate_scale, down_q, down_scale, act: str,
                  active: np.ndarray, perm=None) -> tuple[np.ndarray, np.ndarray]:
    """:func:`ffn_sparse_q8` for 4-bit rows (PowerInfer's OPT-30B-Q4 runs): the
    same weight = code x scale, with every code an int8 in [-8, 7]; the two-
    codes-per-byte storage is an encoding (:func:`pack_q4`), not arithmetic."""
    for q in (up_q, gate_q, down_q):
        if q is not None and (q.min() < -8 or q.max() > 7):
            raise ValueError("4-bit codes must lie in [-8, 7]")
    return ffn_sparse_q8(x, up_q, up_scale, gate_q, gate_scale, down_q, down_scale, act, active, perm)


def pack_q4(codes: np.ndarray) -> np.ndarray:
    """Storage of 4-bit codes along the last axis (even length): byte i holds
    code 2i in its low half and code 2i+1 in its high half, each as a 4-bit
    two's-complement number."""
    c = np.asarray(codes).astype(np.int16)
    lo, hi = c[..., 0::2] & 15, c[..., 1::2] & 15
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_q4(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_q4`: int8 codes in [-8, 7]."""
    b = np.asarray(packed).astype(np.int16)
    lo, hi = b & 15, b >> 4
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int16)
    out[..., 0::2], out[..., 1::2] = lo, hi
    return np.where(out >= 8, out - 16, out).astype(np.int8)


# --------------------------------------------------------------------------
# One layer, one or more tokens
# --------------------------------------------------------------------------

def decode_layer(x: np.ndarray, W1, W2, up, gate, down, act: str, thres: float,
                 group_size: int, perm=None, b1=None, b2=None, active_override=None) -> dict:
    """Predictor, threshold and sparse FFN for one token of one layer.

    All weight arguments are float64 in original neuron order, W2 (f, h) one
    row per ORIGINAL neuron. The predictor's score for slot s is the score of
    neuron perm[s]. ``active_override`` (bool, slot order) replaces the
    predicted mask for the FFN step; the predicted views are still returned.
    """
    f = W2.shape[0]
    if perm is None:
        perm = np.arange(f)
    perm = np.asarray(perm)
    hid = predictor_hidden(W1, x, b1)
    scores_orig = predictor_scores(W2, hid, b2)
    scores = scores_orig[perm]                      # slot order
    active = active_from_scores(scores, thres)
    views = mask_views(active, group_size)
    use = active if active_override is None else np.asarray(active_override, dtype=bool)
    y, h = ffn_sparse(x, up, gate, down, act, use, perm)
    return {"hid": hid, "scores": scores, "active": active, "y": y, "h": h, **views}


def batch_union(actives: np.ndarray, group_size: int) -> dict:
    """Union of a batch's active sets (reading: each token keeps its own mask
    for its own output; the union only decides which rows are loaded and what
    the group-momentum update sees). actives is (B, f) bool in slot order."""
    u = np.asarray(actives, dtype=bool).any(axis=0)
    v = mask_views(u, group_size)
    return {"active": u, "unmask": v["nmask"], "ugmask": v["gmask"],
            "uidx": v["idx"], "ucount": v["count"]}


# --------------------------------------------------------------------------
# Temporal activation momentum (KAIROX 核心方法 item 4) in float32
# --------------------------------------------------------------------------

def tam_threshold(lam: np.float32, eps: np.float32) -> tuple[np.float32, np.float32]:
    """om = 1 - lambda and tau = om + eps, each rounded to float32."""
    lam = np.float32(lam)
    om = np.float32(np.float32(1.0) - lam)
    tau = np.float32(om + np.float32(eps))
    return om, tau


def tam_scores_step(scores: np.ndarray, gactive: np.ndarray, lam, eps) -> tuple[np.ndarray, np.float32]:
    """One momentum step over all groups, float32, one rounding per operation.

    Reading of the page's prose ("accumulates when active, decays by lambda
    when not", with tau = (1 - lambda) + eps "just above the score of one
    isolated activation"): the exponential moving average
        s <- lambda * s + (1 - lambda) * [group active]
    which leaves one isolated hit from rest at exactly 1 - lambda < tau. The
    multiply and the add are rounded separately (no fused multiply-add).
    Returns (new scores, tau).
    """
    lam = np.float32(lam)
    om, tau = tam_threshold(lam, eps)
    s = np.asarray(scores, dtype=np.float32)
    s = (lam * s).astype(np.float32)
    add = np.where(np.asarray(gactive, dtype=bool), om, np.float32(0.0)).astype(np.float32)
    s = (s + add).astype(np.float32)
    return s, tau


def tam_select(scores: np.ndarray, tau: np.float32, capacity_k: int) -> tuple[np.ndarray, np.ndarray]:
    """Candidates are groups with score > tau (strict: the page says the score
    must exceed tau). Of those, the capacity_k highest scores stay resident;
    ties go to the lower group index (a reading; the page names a GPU argsort
    without a tie rule). Returns (cand bool, topk int32 in rank order)."""
    s = np.asarray(scores, dtype=np.float32)
    cand = s > np.float32(tau)
    ids = np.flatnonzero(cand)
    # sort by (-score, index) with a stable sort on the index-ordered list
    order = ids[np.argsort(-s[ids].astype(np.float64), kind="stable")]
    k = max(0, min(int(capacity_k), order.shape[0]))
    return cand, order[:k].astype(np.int32)


def tam_update(scores: np.ndarray, prev_resident: np.ndarray, gactive: np.ndarray,
               lam, eps, capacity_k: int) -> dict:
    """Full per-layer update: new scores, candidate set, resident set, and the
    load/evict/changed sets from the fused AND-NOT / XOR of the bitsets
    (KAIROX 核心方法 item 6): load = res & ~prev, evict = prev & ~res,
    changed = res ^ prev. Bool arrays over groups; words via bits_to_words."""
    n = np.asarray(scores).shape[0]
    s, tau = tam_scores_step(scores, gactive, lam, eps)
    cand, topk = tam_select(s, tau, capacity_k)
    res = np.zeros(n, dtype=bool)
    res[topk] = True
    prev = np.asarray(prev_resident, dtype=bool)
    return {
        "scores": s, "tau": tau, "cand": cand, "n_cand": int(cand.sum()), "topk": topk,
        "resident": res, "load": res & ~prev, "evict": prev & ~res, "changed": res ^ prev,
    }


def tam_closed_form(acts: np.ndarray, lam: float, s0: float = 0.0) -> float:
    """Closed form of the momentum recursion in float64, independent of the
    float32 step: s_T = lambda^T s_0 + (1 - lambda) * sum_t lambda^(T-t) a_t
    for a 0/1 sequence a_1..a_T."""
    a = np.asarray(acts, dtype=np.float64)
    T = a.shape[0]
    pw = np.array([lam ** (T - t) for t in range(1, T + 1)], dtype=np.float64)
    return float(lam ** T * s0 + (1.0 - lam) * np.dot(pw, a))


# --------------------------------------------------------------------------
# Adaptive Neuron Balancer (KAIROX 核心方法 item 5)
# --------------------------------------------------------------------------

def anb_step(lam, stall_io: bool, alpha, lo, hi) -> np.float32:
    """One binary-feedback step of lambda, float32: an I/O stall raises lambda
    by alpha, a compute stall lowers it by alpha, then clamp to [lo, hi]. The
    page names the step size without a value; the caller passes it."""
    lam = np.float32(lam)
    step = np.float32(alpha) if stall_io else np.float32(-np.float32(alpha))
    v = np.float32(lam + step)
    return np.float32(min(np.float32(hi), max(np.float32(lo), v)))


# --------------------------------------------------------------------------
# Dense reference of the same FFN (the all-active special case)
# --------------------------------------------------------------------------

def ffn_dense(x: np.ndarray, up, gate, down, act: str) -> np.ndarray:
    """All neurons computed: y = down @ act(up @ x, gate @ x)."""
    u = up @ x
    g = gate @ x if gate is not None else None
    return down @ activation(act, u, g)


def bits_of(words: np.ndarray, n: int) -> list[int]:
    """Sorted list of set element indices (helper for readable test output)."""
    return [i for i in range(n) if (int(words[i // 32]) >> (i % 32)) & 1]


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "math", "np")]
