"""The seeded generator reproduces the workload statistics it is asked for.

Targets: mean active fraction per token (PowerInfer §3.2 footnote and §8.2;
~50% for SiLU models, §4), top-q coverage (PowerInfer §3.1 Insight 1), batch
union growth (KAIROX 问题与动机: larger batches activate more neurons),
temporal correlation of consecutive tokens, and seed determinism. Scores
are evaluated by the oracle; the generator itself evaluates nothing.
"""

import hashlib

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gb300 import workload as W
from oracle import sffn_oracle as O


def _active_matrix(spec, T, seed=0, d=None):
    if d is not None:
        spec = W.spec_replace(spec, d=d)
    L = W.make_layer(spec, seed=seed, layer=0, with_down=False)
    X = W.spec_tokens(spec, T, seed=seed)
    W1 = O.widen(W.stored_numpy(L["W1"]), spec.wdtype)
    W2 = O.widen(W.stored_numpy(L["W2"]), spec.wdtype)
    b2 = None if L["b2"] is None else L["b2"].numpy().astype(np.float64)
    perm = L["perm"].numpy()
    rows = []
    for t in range(T):
        hid = O.predictor_hidden(W1, X[t, 0].numpy().astype(np.float64))
        rows.append(O.predictor_scores(W2, hid, b2)[perm] >= spec.thres)
    return spec, L, np.array(rows)


@pytest.mark.parametrize("name,d", [
    ("relu_d512_f2048_fp32", None),
    ("opt6.7b_relu_d4096_f16384_fp16", 1024),
    ("llama2_70b_reglu_d8192_f28672_bf16_8l", 1024),
    ("swiglu7b_d4096_f11008_bf16_32l", 1024),
])
def test_active_fraction_and_coverage(name, d):
    spec = W.WORKLOADS[name]
    spec, L, A = _active_matrix(spec, 120, d=d)
    frac = A.mean()
    assert abs(frac - spec.p_mean) < 0.15 * spec.p_mean, frac
    # per-slot empirical frequency follows the planted probability
    assert np.corrcoef(A.mean(0), L["p_slot"])[0, 1] > 0.75
    if spec.coverage is not None:
        freq = np.sort(A.mean(0))[::-1]
        k = int(spec.coverage[0] * spec.f)
        cov = freq[:k].sum() / freq.sum()
        assert abs(cov - spec.coverage[1]) < 0.08, cov


def test_batch_union_grows_to_target():
    spec = W.spec_replace(W.WORKLOADS["falcon40b_relu_d8192_f32768_fp16_batch"], d=1024)
    spec, L, A = _active_matrix(spec, 64)
    unions = [A[:b].any(0).mean() for b in (1, 4, 8, 16, 32)]
    assert all(b > a for a, b in zip(unions, unions[1:])), unions
    assert abs(unions[-1] - spec.union_target[1]) < 0.06, unions
    assert abs(A.mean() - spec.p_mean) < 0.015


def test_groups_coactivate():
    spec = W.WORKLOADS["relu_d512_f2048_fp32"]
    spec, L, A = _active_matrix(spec, 200)
    G = spec.group_size
    # mean pairwise correlation of activity inside a group vs across groups
    X = A.astype(np.float64) - A.mean(0)
    sd = X.std(0) + 1e-12
    C = (X.T @ X) / A.shape[0] / np.outer(sd, sd)
    grp = np.arange(spec.f) // G
    same = (grp[:, None] == grp[None, :]) & ~np.eye(spec.f, dtype=bool)
    busy = A.mean(0) > 0.05
    m = busy[:, None] & busy[None, :]
    assert C[same & m].mean() > C[~same & m].mean() + 0.1


def test_ar1_tokens_correlated():
    X = W.make_tokens(4096, 300, seed=3, kind="ar1")[:, 0].double()
    cos = torch.nn.functional.cosine_similarity(X[1:], X[:-1], dim=1).mean().item()
    assert 0.87 < cos < 0.92          # 0.9 / sqrt(0.81 + 0.44^2) ~ 0.898
    var = X[50:].var().item()
    assert abs(var - 0.1936 / (1 - 0.81)) < 0.05
    Xi = W.make_tokens(512, 100, seed=3, kind="iid")[:, 0].double()
    assert abs(torch.nn.functional.cosine_similarity(Xi[1:], Xi[:-1], dim=1).mean().item()) < 0.05


def test_ar1_variant_at_098_cosine():
    spec = W.WORKLOADS["opt6.7b_relu_d4096_f16384_fp16_rho098"]
    X = W.spec_tokens(spec, 300, seed=3)[:, 0].double()
    cos = torch.nn.functional.cosine_similarity(X[1:], X[:-1], dim=1).mean().item()
    assert 0.975 < cos < 0.985       # 0.98 / sqrt(0.98^2 + 0.199^2) ~ 0.980
    assert abs(X[50:].var().item() - 1.0) < 0.05
    # the base workload's tokens are unchanged by passing its coefficients explicitly
    base = W.WORKLOADS["opt6.7b_relu_d4096_f16384_fp16"]
    assert torch.equal(W.spec_tokens(base, 20, seed=3), W.make_tokens(base.d, 20, seed=3, kind="ar1"))


def test_correlated_tokens_keep_their_active_sets():
    """Consecutive tokens at 0.98 cosine share more of their active set than at
    0.9, at the same mean active fraction."""
    def overlap(name):
        spec, _, A = _active_matrix(W.WORKLOADS[name], 60, d=1024)
        inter = (A[1:] & A[:-1]).sum(1)
        union = (A[1:] | A[:-1]).sum(1)
        return float((inter / np.maximum(union, 1)).mean()), float(A.mean())
    j09, f09 = overlap("opt6.7b_relu_d4096_f16384_fp16")
    j98, f98 = overlap("opt6.7b_relu_d4096_f16384_fp16_rho098")
    assert abs(f98 - f09) < 0.02, (f09, f98)
    assert j98 > j09 + 0.1, (j09, j98)


def test_seed_determinism_and_independence():
    spec = W.WORKLOADS["relu_d512_f2048_fp32"]

    def digest(seed, layer):
        L = W.make_layer(spec, seed=seed, layer=layer)
        h = hashlib.sha256()
        for k in ("W1", "W2", "up", "down", "perm", "b2"):
            h.update(W.stored_numpy(L[k]).tobytes())
        return h.hexdigest()

    assert digest(0, 0) == digest(0, 0)
    assert digest(0, 0) != digest(1, 0)
    assert digest(0, 0) != digest(0, 1)


def test_zipf_solvers():
    p = W.zipf_probs(10000, 1.2, 0.1)
    assert abs(p.mean() - 0.1) < 1e-9 and p.max() <= 0.995 and (np.diff(p) <= 0).all()
    a = W.solve_alpha_coverage(10000, 0.1, 0.26, 0.8)
    p = W.zipf_probs(10000, a, 0.1)
    assert abs(p[:2600].sum() / p.sum() - 0.8) < 1e-6
    a = W.solve_alpha_union(8192, 0.07, 32, 0.4)
    p = W.zipf_probs(8192, a, 0.07)
    assert abs(np.mean(1 - (1 - p) ** 32) - 0.4) < 1e-6


def test_perm_is_permutation_and_stored_dtypes():
    for name in W.WORKLOADS:
        spec = W.spec_replace(W.WORKLOADS[name], d=64, f=256, h=32) if name != "relu_d512_f2048_fp32" else W.WORKLOADS[name]
        if spec.union_target is not None:
            spec = W.spec_replace(spec, union_target=(32, 0.6))
        L = W.make_layer(spec, seed=0, layer=0)
        assert sorted(L["perm"].tolist()) == list(range(spec.f))
        sfx = "_q" if spec.ffn_quant else ""
        assert L["W1"].dtype == W.torch_dtype(spec.wdtype) and L["up" + sfx].shape == (spec.f, spec.d)
        assert L["down" + sfx].shape == (spec.d, spec.f)
        assert (L["gate" + sfx] is None) == (not spec.gated)


def test_stall_bits():
    s = W.make_stall_bits(1024, 32, seed=0)
    assert s.shape == (1024, 32) and s.dtype == np.uint8
    assert abs(s.mean() - 0.5) < 0.02
    assert (s == W.make_stall_bits(1024, 32, seed=0)).all()


def test_quantize_rows_q8():
    g = torch.Generator().manual_seed(0)
    w = torch.randn(64, 48, generator=g).to(torch.bfloat16)
    w[3] = 0.0
    q, s = W.quantize_rows_q8(w)
    assert q.dtype == torch.int8 and s.dtype == torch.float32 and q.shape == w.shape and s.shape == (64,)
    assert int(q.abs().max()) <= 127
    nz = torch.arange(64) != 3
    assert (q[nz].abs().amax(dim=1) == 127).all()          # the largest |w| of a row maps to 127
    assert s[3] == 1.0 and (q[3] == 0).all()
    err = (q.float() * s[:, None] - w.float()).abs()
    assert (err <= s[:, None] / 2 + 1e-7).all()            # rounding to the nearest code


def test_q8_layer_fields():
    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_q8_8l"], d=256, f=512, h=64)
    w = W.make_layer(spec, seed=0)
    assert w["up"] is None and w["gate"] is None and w["down"] is None
    assert w["up_q"].shape == (512, 256) and w["gate_q"].shape == (512, 256) and w["down_q"].shape == (256, 512)
    assert w["up_s"].shape == w["gate_s"].shape == w["down_s"].shape == (512,)
    assert W.WORKLOADS["llama2_70b_reglu_d8192_f28672_q8_8l"].fbytes == 1


def test_quantize_rows_q4():
    g = torch.Generator().manual_seed(1)
    w = torch.randn(40, 64, generator=g).to(torch.bfloat16)
    q, s = W.quantize_rows_q8(w, bits=4)
    assert q.dtype == torch.int8 and int(q.min()) >= -7 and int(q.max()) <= 7
    assert (q.abs().amax(dim=1) == 7).all()                 # the largest |w| of a row maps to 7
    err = (q.float() * s[:, None] - w.float()).abs()
    assert (err <= s[:, None] / 2 + 1e-7).all()


def test_q4_layer_fields():
    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_q4_8l"], d=256, f=512, h=64)
    w = W.make_layer(spec, seed=0)
    assert w["qbits"] == 4 and w["up"] is None and int(w["down_q"].abs().max()) <= 7
    assert spec.fbytes == 0.5 and spec.ffn_quant
