"""Seeded synthetic workloads for the activation-sparse FFN decode step.

This module draws inputs only: weights, token sequences and stall bits. It
evaluates no step of the method (no predictor, no FFN, no momentum update),
so the CUDA path and the CPU oracle can both be fed from it without sharing
any of the method's arithmetic.

Shapes and statistics follow the workloads the pages describe: OPT-, LLaMA2-,
Falcon- and 7B-SwiGLU-shaped FFN layers; power-law activation where a small
share of neurons does most of the firing (PowerInfer §3.1, Insight 1); about
10-20% active per token for ReLU models and about 50% for SiLU models
(PowerInfer §3.2 footnote, §8.2, §4); co-activated neurons stored together in
groups (KAIROX 核心方法 items 1 and 3); temporally correlated tokens
(KAIROX observation 3). Real profiles, trained predictors and datasets are not
available, so these statistics are synthesised:

* Every neuron gets a firing probability from a Zipf law p_r = min(p_max,
  C r^-alpha) over its rank r, with C chosen for the target mean and alpha
  solved for the target coverage ("the top q of neurons give c of the
  activations") or for a target batch-union size.
* Ranks are assigned a group at a time: group g holds G consecutive ranks and
  the group order is a seeded shuffle. This is the layout after co-activation
  reordering.
* Predictor rows of one group share a common component (weight rho), which
  makes their scores co-vary.
* The firing probability is placed with a closed-form Gaussian approximation
  of the predictor score over random inputs: either a per-row offset of W2
  along the all-ones direction (the default; the predictor stays exactly
  W2 . ReLU(W1 . x), which is positively homogeneous in x, so the active set
  depends only on the direction of x), or an output bias b2 (used by the tiny
  single-layer workload, whose description asks for a bias).
"""

from __future__ import annotations

import dataclasses
import hashlib
import math

import numpy as np
import torch

# ReLU of a standard normal: mean and variance
_RELU_MEAN = 1.0 / math.sqrt(2.0 * math.pi)
_RELU_VAR = 0.5 - 1.0 / (2.0 * math.pi)


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and activation statistics of one synthetic FFN layer."""

    name: str
    d: int                      # model dimension
    f: int                      # FFN neurons
    h: int                      # predictor hidden size
    group_size: int             # co-activation group size G
    act: str                    # "relu" | "reglu" | "swiglu" | "relu2" (squared ReLU)
    wdtype: str                 # "f32" | "f16" | "bf16"
    p_mean: float               # mean firing probability per token
    zipf_alpha: float | None = None          # fixed alpha, or
    coverage: tuple | None = None            # (top fraction, share of activations), or
    union_target: tuple | None = None        # (batch size, mean union fraction)
    p_max: float = 0.995
    rho_group: float = 0.5      # shared component of predictor rows in a group
    bias_mode: bool = False     # place p with b2 instead of a W2 row offset
    layers: int = 1
    tokens: int = 64
    seq: str = "iid"            # "iid" | "ar1"
    ar_rho: float = 0.9
    ar_noise: float = 0.44
    batches: tuple = (1,)
    thres: float = 0.0
    tam_lambda: float = 0.9
    tam_eps: float = 0.01
    tam_capacity: int | None = None          # default: half of the groups
    anb: bool = False
    anb_alpha: float = 0.01
    anb_lo: float = 0.8
    anb_hi: float = 0.99
    topic_shift_at: int | None = None
    ffn_q8: bool = False        # FFN rows as 8-bit codes with one scale per neuron (predictor stays wdtype)
    ffn_q4: bool = False        # the same with 4-bit codes (two per stored byte)

    @property
    def n_groups(self) -> int:
        return self.f // self.group_size

    @property
    def capacity(self) -> int:
        return self.tam_capacity if self.tam_capacity is not None else self.n_groups // 2

    @property
    def wbytes(self) -> int:
        return {"f32": 4, "f16": 2, "bf16": 2}[self.wdtype]

    @property
    def fbytes(self) -> float:
        """Bytes per stored FFN weight (0.5 for 4-bit codes)."""
        return 0.5 if self.ffn_q4 else 1 if self.ffn_q8 else self.wbytes

    @property
    def ffn_quant(self) -> bool:
        """FFN rows stored as codes with one scale per neuron (8-bit or 4-bit)."""
        return self.ffn_q8 or self.ffn_q4

    @property
    def n_mats(self) -> int:
        return 3 if self.gated else 2

    @property
    def gated(self) -> bool:
        """ReGLU and SwiGLU read a gate row per neuron; ReLU and squared ReLU do not."""
        return self.act in ("reglu", "swiglu")


# The workloads, named by what they are.
WORKLOADS = {
    # Tiny single ReLU layer: fp32, Zipf(1.1) ranks, ~10% active via b2.
    "relu_d512_f2048_fp32": LayerSpec(
        name="relu_d512_f2048_fp32", d=512, f=2048, h=64, group_size=32, act="relu",
        wdtype="f32", p_mean=0.10, zipf_alpha=1.1, bias_mode=True, tokens=64, seq="iid",
        tam_capacity=32),
    # OPT-6.7B-shaped ReLU layer, fp16, ~8% active, top 20% -> 80%.
    "opt6.7b_relu_d4096_f16384_fp16": LayerSpec(
        name="opt6.7b_relu_d4096_f16384_fp16", d=4096, f=16384, h=1024, group_size=32,
        act="relu", wdtype="f16", p_mean=0.08, coverage=(0.20, 0.80), tokens=256, seq="ar1"),
    # The same layer with consecutive tokens at ~0.98 cosine: rho 0.98 with noise
    # 0.199 keeps unit variance (0.98^2 + 0.199^2 = 1.0).
    "opt6.7b_relu_d4096_f16384_fp16_rho098": LayerSpec(
        name="opt6.7b_relu_d4096_f16384_fp16_rho098", d=4096, f=16384, h=1024, group_size=32,
        act="relu", wdtype="f16", p_mean=0.08, coverage=(0.20, 0.80), tokens=256, seq="ar1",
        ar_rho=0.98, ar_noise=0.199),
    # LLaMA2-70B-shaped ReGLU stack, bf16, 8 layers, ~10% active, top 26% -> 80%.
    "llama2_70b_reglu_d8192_f28672_bf16_8l": LayerSpec(
        name="llama2_70b_reglu_d8192_f28672_bf16_8l", d=8192, f=28672, h=1024, group_size=64,
        act="reglu", wdtype="bf16", p_mean=0.10, coverage=(0.26, 0.80), layers=8, tokens=512,
        seq="ar1", tam_capacity=224),
    # The same stack with 8-bit FFN rows (the quantized variant; bf16 predictor).
    "llama2_70b_reglu_d8192_f28672_q8_8l": LayerSpec(
        name="llama2_70b_reglu_d8192_f28672_q8_8l", d=8192, f=28672, h=1024, group_size=64,
        act="reglu", wdtype="bf16", p_mean=0.10, coverage=(0.26, 0.80), layers=8, tokens=512,
        seq="ar1", tam_capacity=224, ffn_q8=True),
    # ... and with 4-bit FFN rows (PowerInfer runs OPT-30B at Q4).
    "llama2_70b_reglu_d8192_f28672_q4_8l": LayerSpec(
        name="llama2_70b_reglu_d8192_f28672_q4_8l", d=8192, f=28672, h=1024, group_size=64,
        act="reglu", wdtype="bf16", p_mean=0.10, coverage=(0.26, 0.80), layers=8, tokens=512,
        seq="ar1", tam_capacity=224, ffn_q4=True),
    # Falcon-40B-shaped ReLU layer under batching, fp16, ~7% per token, union ~40% at B=32.
    "falcon40b_relu_d8192_f32768_fp16_batch": LayerSpec(
        name="falcon40b_relu_d8192_f32768_fp16_batch", d=8192, f=32768, h=1024, group_size=32,
        act="relu", wdtype="f16", p_mean=0.07, union_target=(32, 0.40), tokens=64, seq="iid",
        batches=(1, 4, 8, 16, 32)),
    # 7B-shaped SwiGLU decode loop, bf16, 32 layers, ~50% active, top 69% -> 80%,
    # adaptive lambda, topic shift half way.
    "swiglu7b_d4096_f11008_bf16_32l": LayerSpec(
        name="swiglu7b_d4096_f11008_bf16_32l", d=4096, f=11008, h=512, group_size=32,
        act="swiglu", wdtype="bf16", p_mean=0.50, coverage=(0.69, 0.80), layers=32,
        tokens=1024, seq="ar1", anb=True, topic_shift_at=512),
}


def spec_replace(spec: LayerSpec, **kw) -> LayerSpec:
    """A copy of ``spec`` with some fields changed (e.g. smaller shapes)."""
    return dataclasses.replace(spec, **kw)


# --------------------------------------------------------------------------
# Seeds
# --------------------------------------------------------------------------

def sub_seed(seed: int, *keys) -> int:
    """A 63-bit seed derived from ``seed`` and a tuple of keys (SHA-256)."""
    h = hashlib.sha256(repr((int(seed),) + tuple(keys)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int, *keys) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, *keys))
    return g


# --------------------------------------------------------------------------
# Zipf firing probabilities
# --------------------------------------------------------------------------

def zipf_probs(n: int, alpha: float, p_mean: float, p_max: float = 0.995) -> np.ndarray:
    """p_r = min(p_max, C r^-alpha), r = 1..n, with C chosen so mean(p) = p_mean."""
    r = np.arange(1, n + 1, dtype=np.float64)
    base = r ** (-alpha)
    lo, hi = 0.0, p_max / base[-1] * 2.0
    for _ in range(200):
        c = 0.5 * (lo + hi)
        if np.minimum(p_max, c * base).mean() < p_mean:
            lo = c
        else:
            hi = c
    return np.minimum(p_max, 0.5 * (lo + hi) * base)


def _bisect_alpha(fn, target: float, lo: float = 0.0, hi: float = 6.0) -> float:
    """alpha with fn(alpha) = target for fn increasing in alpha."""
    for _ in range(80):
        mid = 0.5 * (lo + hi)
        if fn(mid) < target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def solve_alpha_coverage(n: int, p_mean: float, top_frac: float, share: float, p_max: float = 0.995) -> float:
    """alpha such that the top ``top_frac`` of neurons give ``share`` of the
    expected activations (PowerInfer §3.1, Insight 1)."""
    k = max(1, int(round(top_frac * n)))

    def cov(a):
        p = zipf_probs(n, a, p_mean, p_max)
        return p[:k].sum() / p.sum()

    return _bisect_alpha(cov, share)


def solve_alpha_union(n: int, p_mean: float, batch: int, target: float, p_max: float = 0.995) -> float:
    """alpha such that the expected fraction of neurons active for at least one
    of ``batch`` independent tokens is ``target`` (more skew, smaller union)."""

    def neg_union(a):
        p = zipf_probs(n, a, p_mean, p_max)
        return -np.mean(1.0 - (1.0 - p) ** batch)

    return _bisect_alpha(neg_union, -target)


def spec_alpha(spec: LayerSpec) -> float:
    if spec.zipf_alpha is not None:
        return spec.zipf_alpha
    if spec.coverage is not None:
        return solve_alpha_coverage(spec.f, spec.p_mean, spec.coverage[0], spec.coverage[1], spec.p_max)
    if spec.union_target is not None:
        return solve_alpha_union(spec.f, spec.p_mean, spec.union_target[0], spec.union_target[1], spec.p_max)
    return 0.0


def slot_probabilities(spec: LayerSpec, seed: int, layer: int, topic: int = 0) -> np.ndarray:
    """Firing probability of every packed slot. Group g gets the block of
    consecutive ranks at a seeded position; topic != 0 redraws that order."""
    p_rank = zipf_probs(spec.f, spec_alpha(spec), spec.p_mean, spec.p_max)
    rng = np.random.default_rng(sub_seed(seed, "group_rank", layer, topic))
    grank = rng.permutation(spec.n_groups)
    G = spec.group_size
    ranks = (grank[:, None] * G + np.arange(G)[None, :]).reshape(-1)
    return p_rank[ranks]


# --------------------------------------------------------------------------
# Layers
# --------------------------------------------------------------------------

_TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def torch_dtype(wdtype: str) -> torch.dtype:
    return _TORCH_DTYPE[wdtype]


def _normal(shape, std, gen, device):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32) * std


def _ndtri(p: torch.Tensor) -> torch.Tensor:
    return torch.special.ndtri(p.to(torch.float64))


def _row_offsets(z: torch.Tensor, c: torch.Tensor, q: torch.Tensor) -> torch.Tensor:
    """Offsets beta (one per row of z) such that, for r_j iid ReLU(N(0,1)),
    the Gaussian approximation of sum_j c_j (z_j + beta) r_j has
    mean / std = q. Shaping arithmetic of the generator only."""
    z = z.to(torch.float64)
    c = c.to(torch.float64)
    k = q * math.sqrt(_RELU_VAR) / _RELU_MEAN
    S = z @ c
    T = c.sum()
    Q = (z * z) @ (c * c)
    R = z @ (c * c)
    U = (c * c).sum()
    a = T * T - k * k * U
    b = 2.0 * (S * T - k * k * R)
    cc = S * S - k * k * Q
    disc = torch.clamp(b * b - 4.0 * a * cc, min=0.0)
    r1 = (-b + torch.sqrt(disc)) / (2.0 * a)
    r2 = (-b - torch.sqrt(disc)) / (2.0 * a)
    ok1 = torch.sign(S + r1 * T) == torch.sign(k)
    beta = torch.where(ok1, r1, r2)
    return torch.where(k == 0, -S / T, beta)


def make_layer(spec: LayerSpec, seed: int = 0, layer: int = 0, device="cpu", topic: int = 0,
               with_down: bool = True) -> dict:
    """Draw one layer's weights in the stored dtype, in ORIGINAL neuron order.

    Returns W1 (h, d), W2 (f, h), up (f, d), gate (f, d) or None, down (d, f),
    perm (f,) int32 with perm[slot] = original neuron id, b1/b2 (float32 or
    None) and p_slot (firing probabilities by slot, float64 numpy).
    """
    d, f, h, G = spec.d, spec.f, spec.h, spec.group_size
    dt = torch_dtype(spec.wdtype)
    W1 = _normal((h, d), 1.0 / math.sqrt(d), _gen(device, seed, "W1", layer), device)
    W1s = W1.to(dt)
    # norms of the stored W1 rows set the scale of each hidden unit
    c = W1s.to(torch.float32).norm(dim=1)
    p_slot = slot_probabilities(spec, seed, layer, topic)
    q = _ndtri(torch.as_tensor(p_slot, device=device))
    gz = _gen(device, seed, "W2z", layer)
    u = _normal((spec.n_groups, h), 1.0, gz, device)
    v = _normal((f, h), 1.0, gz, device)
    z = math.sqrt(spec.rho_group) * u.repeat_interleave(G, dim=0) + math.sqrt(1.0 - spec.rho_group) * v
    b2 = None
    if spec.bias_mode:
        W2_slot = z / math.sqrt(h)
        zz = W2_slot.to(dt).to(torch.float64)
        mean = _RELU_MEAN * (zz @ c.to(torch.float64))
        std = torch.sqrt(_RELU_VAR * ((zz * zz) @ (c.to(torch.float64) ** 2)))
        b2_slot = (q * std - mean).to(torch.float32)
    else:
        beta = _row_offsets(z, c, q)
        W2_slot = ((z.to(torch.float64) + beta[:, None]) / math.sqrt(h)).to(torch.float32)
    rng = np.random.default_rng(sub_seed(seed, "perm", layer))
    perm_np = rng.permutation(f).astype(np.int32)
    perm = torch.as_tensor(perm_np, device=device)
    W2 = torch.empty((f, h), dtype=torch.float32, device=device)
    W2[perm.long()] = W2_slot
    if spec.bias_mode:
        b2 = torch.empty(f, dtype=torch.float32, device=device)
        b2[perm.long()] = b2_slot
    up = _normal((f, d), 1.0 / math.sqrt(d), _gen(device, seed, "up", layer), device).to(dt)
    gate = None
    if spec.gated:
        gate = _normal((f, d), 1.0 / math.sqrt(d), _gen(device, seed, "gate", layer), device).to(dt)
    down = None
    if with_down:
        down = _normal((d, f), 1.0 / math.sqrt(f), _gen(device, seed, "down", layer), device).to(dt)
    w = {
        "W1": W1s, "W2": W2.to(dt), "b1": None, "b2": b2, "up": up, "gate": gate, "down": down,
        "perm": perm, "p_slot": p_slot,
    }
    if spec.ffn_q4:
        return quantize_layer_q8(w, bits=4)
    return quantize_layer_q8(w) if spec.ffn_q8 else w


def make_w2_topic(spec: LayerSpec, seed: int, layer: int, topic: int, W1: torch.Tensor,
                  perm: torch.Tensor) -> torch.Tensor:
    """W2 of ``layer`` after a topic shift: same shared/independent row
    components, offsets re-placed for the redrawn group ranks."""
    device = W1.device
    dt = torch_dtype(spec.wdtype)
    h, G = spec.h, spec.group_size
    c = W1.to(torch.float32).norm(dim=1)
    p_slot = slot_probabilities(spec, seed, layer, topic)
    q = _ndtri(torch.as_tensor(p_slot, device=device))
    gz = _gen(device, seed, "W2z", layer)
    u = _normal((spec.n_groups, h), 1.0, gz, device)
    v = _normal((spec.f, h), 1.0, gz, device)
    z = math.sqrt(spec.rho_group) * u.repeat_interleave(G, dim=0) + math.sqrt(1.0 - spec.rho_group) * v
    beta = _row_offsets(z, c, q)
    W2_slot = ((z.to(torch.float64) + beta[:, None]) / math.sqrt(h)).to(torch.float32)
    W2 = torch.empty_like(W2_slot)
    W2[perm.long()] = W2_slot
    return W2.to(dt)


def make_tokens(d: int, T: int, seed: int = 0, kind: str = "iid", batch: int = 1,
                ar_rho: float = 0.9, ar_noise: float = 0.44, device="cpu", stream: int = 0) -> torch.Tensor:
    """Token inputs x, float32, shape (T, batch, d). ``iid``: x ~ N(0, I).
    ``ar1``: x_0 ~ N(0, I), x_{t+1} = ar_rho x_t + ar_noise e_t with e_t ~ N(0, I)
    (one independent sequence per batch row)."""
    g = _gen(device, seed, "tokens", kind, batch, stream)
    e = torch.randn(T, batch, d, generator=g, device=device, dtype=torch.float32)
    if kind == "iid":
        return e
    if kind != "ar1":
        raise ValueError(kind)
    x = torch.empty_like(e)
    x[0] = e[0]
    for t in range(1, T):
        x[t] = ar_rho * x[t - 1] + ar_noise * e[t]
    return x


def spec_tokens(spec: LayerSpec, T: int, seed: int = 0, batch: int = 1, device="cpu") -> torch.Tensor:
    """:func:`make_tokens` with the workload's sequence kind and AR(1) coefficients."""
    return make_tokens(spec.d, T, seed=seed, kind=spec.seq, batch=batch, ar_rho=spec.ar_rho,
                       ar_noise=spec.ar_noise, device=device)


def make_stall_bits(T: int, L: int, seed: int = 0) -> np.ndarray:
    """Seeded binary stall signal per (token, layer): 1 = I/O stall, 0 =
    compute stall, each with probability 1/2."""
    rng = np.random.default_rng(sub_seed(seed, "stall", T, L))
    return rng.integers(0, 2, size=(T, L), dtype=np.uint8)


# --------------------------------------------------------------------------
# Host views of stored tensors (for the oracle)
# --------------------------------------------------------------------------

def quantize_rows_q8(w: torch.Tensor, bits: int = 8) -> tuple[torch.Tensor, torch.Tensor]:
    """Symmetric codes with one float32 scale per row: with m = 2^(bits-1) - 1
    (127 for 8 bits, 7 for 4 bits), scale = max|w| / m (1 for an all-zero
    row), code = round(w / scale), which lies in [-m, m]; int8 either way."""
    m = float(2 ** (bits - 1) - 1)
    wf = w.float()
    amax = wf.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / m, torch.ones_like(amax))
    q = torch.clamp(torch.round(wf / scale[:, None]), -m, m).to(torch.int8)
    return q.contiguous(), scale.contiguous()


def quantize_layer_q8(w: dict, bits: int = 8) -> dict:
    """The layer's FFN rows as 8-bit (or 4-bit) codes: up and gate one scale per
    neuron row, down one scale per neuron column. Returns a new dict with
    up_q/up_s, gate_q/gate_s, down_q/down_s, qbits, and up/gate/down set to None."""
    out = dict(w)
    out["qbits"] = bits
    out["up_q"], out["up_s"] = quantize_rows_q8(w["up"], bits)
    out["gate_q"], out["gate_s"] = quantize_rows_q8(w["gate"], bits) if w.get("gate") is not None else (None, None)
    if w.get("down") is not None:
        qt, s = quantize_rows_q8(w["down"].t(), bits)
        out["down_q"], out["down_s"] = qt.t().contiguous(), s
    out["up"] = out["gate"] = out["down"] = None
    return out


def stored_numpy(t: torch.Tensor | None):
    """The stored bits of a tensor as numpy, in the form the oracle's
    ``widen`` expects: float32, float16, or uint16 patterns for bfloat16."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
