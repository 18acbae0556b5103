"""Shared helpers of the GPU parity tests: host copies of stored weights, the
oracle's view of one token, and the comparisons with their tolerances.

Tolerances of y (see the design notes for the derivation):
  * 16-bit weights, fp32 accumulation: max-abs <= 2e-2 and relative L2 <=
    5e-3 (the stated bar), plus a regression bound of relative L2 <= 1e-4 that
    a pure fp32 rounding difference stays far below (observed ~1e-6).
  * fp32 weights: max-abs <= 1e-4 and relative L2 <= 1e-5.
Mask views are bit-exact except for neurons whose fp64 score lies within
1e-3 of the threshold, which are excluded and counted.
"""

from __future__ import annotations

import numpy as np
import torch

from activation_sparse_ffn_gb300 import workload as W
from oracle import sffn_oracle as O

BAND = 1e-3
TOL = {
    "f32": dict(max_abs=1e-4, rel_l2=1e-5, reg_rel_l2=1e-5),
    "f16": dict(max_abs=2e-2, rel_l2=5e-3, reg_rel_l2=1e-4),
    "bf16": dict(max_abs=2e-2, rel_l2=5e-3, reg_rel_l2=1e-4),
}


def words_bits(words, n: int) -> np.ndarray:
    """Unpack uint32 words (bit i%32 of word i//32) into n bools."""
    w = np.asarray(words).astype(np.uint32).reshape(-1)
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool).reshape(-1)
    return bits[:n]


class HostLayer:
    """Stored (bit-exact) host copies of one layer's weights, original order."""

    def __init__(self, w: dict, wdtype: str):
        self.dt = wdtype
        self.W1 = O.widen(W.stored_numpy(w["W1"]), wdtype)
        self.W2 = O.widen(W.stored_numpy(w["W2"]), wdtype)
        self.q8 = w.get("up_q") is not None     # 8-bit or 4-bit FFN rows: codes and per-neuron scales
        self.qbits = w.get("qbits", 8) if self.q8 else 0
        if self.q8:
            self.q = {k: (w[k].cpu().numpy() if w.get(k) is not None else None)
                      for k in ("up_q", "up_s", "gate_q", "gate_s", "down_q", "down_s")}
            self.up = self.gate = self.down = None
        else:
            self.up = W.stored_numpy(w["up"])
            self.gate = W.stored_numpy(w["gate"]) if w.get("gate") is not None else None
            self.down = W.stored_numpy(w["down"])
        self.perm = w["perm"].cpu().numpy().astype(np.int64) if w.get("perm") is not None else None
        self.b1 = None if w.get("b1") is None else w["b1"].double().cpu().numpy()
        self.b2 = None if w.get("b2") is None else w["b2"].double().cpu().numpy()
        self.f = self.W2.shape[0]

    def scores(self, x: np.ndarray) -> np.ndarray:
        """Predictor scores in slot order, fp64."""
        hid = O.predictor_hidden(self.W1, x, self.b1)
        s = O.predictor_scores(self.W2, hid, self.b2)
        return s if self.perm is None else s[self.perm]

    def ffn(self, x: np.ndarray, active_slots: np.ndarray, act: str) -> np.ndarray:
        if self.q8:
            q = self.q
            fn = O.ffn_sparse_q4 if self.qbits == 4 else O.ffn_sparse_q8
            y, _ = fn(x, q["up_q"], q["up_s"], q["gate_q"], q["gate_s"], q["down_q"], q["down_s"], act,
                      active_slots, self.perm)
            return y
        y, _ = O.ffn_sparse_stored(x, self.up, self.gate, self.down, self.dt, act, active_slots, self.perm)
        return y


def check_masks(scores, thres, G, nmask, gmask, idx, count) -> dict:
    """Compare one token's GPU mask views with the oracle scores."""
    f = scores.shape[0]
    gb = words_bits(nmask, f)
    ob = O.active_from_scores(scores, thres)
    band = np.abs(scores - thres) < BAND
    bad = (gb != ob) & ~band
    assert not bad.any(), f"{bad.sum()} mask bits differ outside the band, e.g. slot {np.flatnonzero(bad)[:5]}"
    # the other views must be exactly the views of the GPU's own bits
    c = int(count)
    assert c == int(gb.sum())
    assert np.array_equal(np.asarray(idx)[:c], np.flatnonzero(gb))
    ng = f // G
    ggb = words_bits(gmask, ng)
    assert np.array_equal(ggb, gb.reshape(ng, G).any(axis=1))
    # and against the oracle for groups that do not hinge on band neurons
    sure_on = (ob & ~band).reshape(ng, G).any(axis=1)
    sure_off = (~ob & ~band).reshape(ng, G).all(axis=1)
    assert not (sure_on & ~ggb).any() and not (sure_off & ggb).any()
    return {"band": int(band.sum()), "active": c, "mismatch_in_band": int(((gb != ob) & band).sum())}


def check_y(y_gpu, y_ref, wdtype: str, what: str = "y") -> dict:
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    nref = np.linalg.norm(y_ref)
    rel = np.linalg.norm(y_gpu - y_ref) / nref if nref > 0 else np.linalg.norm(y_gpu)
    t = TOL[wdtype]
    assert err.max() <= t["max_abs"], f"{what}: max-abs {err.max():.3e} > {t['max_abs']}"
    assert rel <= t["rel_l2"], f"{what}: rel-L2 {rel:.3e} > {t['rel_l2']}"
    assert rel <= t["reg_rel_l2"], f"{what}: rel-L2 {rel:.3e} above the regression bound {t['reg_rel_l2']}"
    return {"max_abs": float(err.max()), "rel_l2": float(rel)}


def make_layer(spec, seed=0, layer=0, max_batch=1, biases=False):
    """Draw a layer on the GPU and pack it; returns (Layer, weights, HostLayer)."""
    from activation_sparse_ffn_gb300 import sffn
    w = W.make_layer(spec, seed=seed, layer=layer, device="cuda")
    if biases:
        g = torch.Generator(device="cuda")
        g.manual_seed(W.sub_seed(seed, "bias", layer))
        w["b1"] = 0.1 * torch.randn(spec.h, generator=g, device="cuda")
        w["b2"] = 0.05 * torch.randn(spec.f, generator=g, device="cuda")
    L = sffn.Layer.from_weights(w, spec.group_size, spec.act, max_batch=max_batch)
    return L, w, HostLayer(w, spec.wdtype)
