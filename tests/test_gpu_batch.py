"""Batched decode (B > 1) against the oracle, through the C ABI.

Each token keeps its own predicted mask for its own output; the union of the
batch's masks decides which rows are read and is reported as union views.
Per-token masks are compared bit-exactly outside the score band, each
token's y against the oracle FFN on that token's own GPU mask (teacher
forcing), and the union views against the OR of the token masks.
"""

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gb300 import workload as W
from oracle import sffn_oracle as O

from gpu_util import check_masks, check_y, make_layer, words_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn as mod
    return mod


def _run(sffn, L, X, thres, x_out=False):
    B = X.shape[0]
    masks = L.masks(B)
    ws = L.workspace(B)
    y = torch.full((B, L.d), float("nan"), device="cuda")
    xo = torch.empty(B, L.d, device="cuda") if x_out else None
    sffn.sffn_decode_step(L.handle, X, B, thres, masks, y, xo, ws)
    torch.cuda.synchronize()
    return masks, y, xo


def _check_batch(host, spec, X, thres, masks, y):
    B = X.shape[0]
    f, G = spec.f, spec.group_size
    union = np.zeros(f, dtype=bool)
    for b in range(B):
        xs = X[b].double().cpu().numpy()
        s = host.scores(xs)
        check_masks(s, thres, G, masks.nmask[b].cpu().numpy(), masks.gmask[b].cpu().numpy(),
                    masks.idx[b].cpu().numpy(), masks.count[b].item())
        gb = words_bits(masks.nmask[b].cpu().numpy(), f)
        union |= gb
        check_y(y[b].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype, f"y[{b}]")
    assert np.array_equal(words_bits(masks.unmask.cpu().numpy(), f), union)
    uc = masks.ucount.item()
    assert uc == int(union.sum())
    assert np.array_equal(masks.uidx[:uc].cpu().numpy(), np.flatnonzero(union))
    ng = f // G
    assert np.array_equal(words_bits(masks.ugmask.cpu().numpy(), ng), union.reshape(ng, G).any(axis=1))


SHAPES = [
    # d, f, h, G, act, dtype. The down product stages 4, 2 or 1 output tiles of
    # 128 per K block depending on d / 128 (8, 16 -> 4; 6 -> 2; 3 -> 1); the
    # contiguous products stage 4 K blocks when h (or d) is a multiple of 256.
    (1024, 2048, 128, 32, "relu", "f16"),
    (1024, 4096, 256, 64, "reglu", "bf16"),
    (2048, 2048, 64, 32, "swiglu", "bf16"),
    (768, 2048, 192, 64, "reglu", "f16"),
    (384, 1024, 64, 32, "relu", "bf16"),
    (1024, 2048, 128, 64, "relu2", "f16"),
    # the views cut each list into four slices of whole group-mask words: a
    # ragged last slice (224 words in slices of 64) and a last group-mask word
    # with one group (65 groups of 32)
    (1024, 7168, 128, 64, "reglu", "bf16"),
    (512, 2080, 64, 32, "relu", "f16"),
]


@pytest.mark.parametrize("d,f,h,G,act,dt", SHAPES)
@pytest.mark.parametrize("B", [2, 5, 16, 17, 32])
def test_batch_matches_oracle(sffn, d, f, h, G, act, dt, B):
    spec = W.LayerSpec(name="t", d=d, f=f, h=h, group_size=G, act=act, wdtype=dt, p_mean=0.12, zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=B, max_batch=32, biases=(B == 5))
    L.set_batch_path("tensor")          # the tensor-core products at every B (auto takes B = 2 to CUDA cores)
    X = W.make_tokens(d, 1, seed=B, batch=B, device="cuda")[0]
    masks, y, _ = _run(sffn, L, X, 0.0)
    _check_batch(host, spec, X, 0.0, masks, y)
    L.check_error()


def test_auto_path_at_two_tokens(sffn):
    """The default choice at B = 2 (the CUDA-core arm on 16-bit rows) against the oracle."""
    spec = W.LayerSpec(name="t", d=2048, f=4096, h=256, group_size=64, act="reglu", wdtype="bf16", p_mean=0.12,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=31, max_batch=32)
    assert sffn.sffn_layer_batch_arm(L.handle, 2) == "cuda_cores"
    assert sffn.sffn_layer_batch_arm(L.handle, 3) == "tensor"
    assert sffn.sffn_layer_batch_arm(L.handle, 1) is None
    X = W.make_tokens(spec.d, 1, seed=32, batch=2, device="cuda")[0]
    masks, y, _ = _run(sffn, L, X, 0.0)
    _check_batch(host, spec, X, 0.0, masks, y)
    L.check_error()


def test_batch_equals_single_calls(sffn):
    spec = W.LayerSpec(name="t", d=1024, f=4096, h=128, group_size=32, act="reglu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.1)
    L, w, host = make_layer(spec, seed=3, max_batch=32)
    X = W.make_tokens(spec.d, 1, seed=4, batch=24, device="cuda")[0]
    masks, y, _ = _run(sffn, L, X, 0.0)
    ws1 = L.workspace(1)
    for b in range(X.shape[0]):
        m1 = L.masks(1)
        y1 = torch.empty(1, spec.d, device="cuda")
        sffn.sffn_decode_step(L.handle, X[b:b + 1], 1, 0.0, m1, y1, None, ws1)
        torch.cuda.synchronize()
        # the two paths round differently, so a neuron may only flip inside the score band
        s = host.scores(X[b].double().cpu().numpy())
        band = np.abs(s) < 1e-3
        diff = words_bits(m1.nmask[0].cpu().numpy(), spec.f) != words_bits(masks.nmask[b].cpu().numpy(), spec.f)
        assert not (diff & ~band).any()
        if not diff.any():
            check_y(y[b].cpu().numpy(), y1[0].double().cpu().numpy(), "bf16", f"batch vs single [{b}]")


def test_identical_tokens_give_the_single_mask(sffn):
    spec = W.LayerSpec(name="t", d=1024, f=2048, h=128, group_size=64, act="swiglu", wdtype="f16", p_mean=0.2,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=5, max_batch=32)
    x = W.make_tokens(spec.d, 1, seed=6, device="cuda")[0]
    X = x.repeat(16, 1).contiguous()
    masks, y, _ = _run(sffn, L, X, 0.0)
    assert torch.equal(masks.unmask, masks.nmask[0])
    for b in range(1, 16):
        assert torch.equal(masks.nmask[b], masks.nmask[0])
        assert torch.equal(y[b], y[0])


def test_batch_forward_with_caller_masks_and_residual(sffn):
    spec = W.LayerSpec(name="t", d=1024, f=2048, h=128, group_size=32, act="relu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=7, max_batch=32)
    B = 8
    rng = np.random.default_rng(8)
    bits = rng.random((B, spec.f)) < np.array([0.0, 1.0, 0.001, 0.05, 0.3, 0.5, 0.02, 0.9])[:, None]
    masks = L.masks(B)
    masks.nmask.copy_(torch.from_numpy(np.stack([O.bits_to_words(b).view(np.int32) for b in bits])).cuda())
    X = W.make_tokens(spec.d, 1, seed=9, batch=B, device="cuda")[0]
    y = torch.empty(B, spec.d, device="cuda")
    xo = torch.empty(B, spec.d, device="cuda")
    sffn.sffn_forward(L.handle, X, B, masks, y, xo, L.workspace(B))
    torch.cuda.synchronize()
    for b in range(B):
        check_y(y[b].cpu().numpy(), host.ffn(X[b].double().cpu().numpy(), bits[b], "relu"), "bf16", f"y[{b}]")
    assert torch.equal(xo, X + y)
    assert (y[0] == 0).all()
    # the union views, formed here from the caller's masks
    union = bits.any(axis=0)
    assert np.array_equal(words_bits(masks.unmask.cpu().numpy(), spec.f), union)
    uc = masks.ucount.item()
    assert uc == int(union.sum())
    assert np.array_equal(masks.uidx[:uc].cpu().numpy(), np.flatnonzero(union))
    ng = spec.f // spec.group_size
    assert np.array_equal(words_bits(masks.ugmask.cpu().numpy(), ng), union.reshape(ng, -1).any(axis=1))
    L.check_error()


def test_batch_predict_views(sffn):
    spec = W.LayerSpec(name="t", d=1024, f=2048, h=128, group_size=32, act="relu", wdtype="f16", p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=10, max_batch=32)
    X = W.make_tokens(spec.d, 1, seed=11, batch=12, device="cuda")[0]
    m1 = L.masks(12)
    sffn.sffn_predict(L.handle, X, 12, 0.0, m1, L.workspace(12))
    m2, y, _ = _run(sffn, L, X, 0.0)
    for k in ("nmask", "gmask", "count", "unmask", "ugmask", "ucount"):
        assert torch.equal(getattr(m1, k), getattr(m2, k)), k


@pytest.mark.parametrize("B", [4, 32])
def test_full_size_falcon_batch(sffn, B):
    spec = W.WORKLOADS["falcon40b_relu_d8192_f32768_fp16_batch"]
    L, w, host = make_layer(spec, seed=0, max_batch=32)
    X = W.make_tokens(spec.d, 1, seed=0, batch=B, device="cuda")[0]
    masks, y, _ = _run(sffn, L, X, spec.thres)
    # every token's mask; y for a sample of tokens (the oracle FFN is the slow part)
    f = spec.f
    union = np.zeros(f, dtype=bool)
    for b in range(B):
        xs = X[b].double().cpu().numpy()
        check_masks(host.scores(xs), spec.thres, spec.group_size, masks.nmask[b].cpu().numpy(),
                    masks.gmask[b].cpu().numpy(), masks.idx[b].cpu().numpy(), masks.count[b].item())
        gb = words_bits(masks.nmask[b].cpu().numpy(), f)
        union |= gb
        if b in (0, B - 1):
            check_y(y[b].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype, f"y[{b}]")
    assert masks.ucount.item() == int(union.sum())
    L.check_error()


def test_fp32_batch_is_unsupported(sffn):
    spec = W.WORKLOADS["relu_d512_f2048_fp32"]
    w = W.make_layer(spec, seed=0, device="cuda")
    L = sffn.Layer.from_weights(w, spec.group_size, spec.act, max_batch=4)
    X = torch.zeros(4, spec.d, device="cuda")
    y = torch.empty(4, spec.d, device="cuda")
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_decode_step(L.handle, X, 4, 0.0, L.masks(4), y, None, L.workspace(1))
    assert e.value.status == sffn.SFFN_ERR_UNSUPPORTED


# ------------------------------------------------------------------ the CUDA-core arm (2 <= B <= 4)

CC_SHAPES = [s for s in SHAPES] + [(8192, 4096, 1024, 64, "reglu", "bf16"), (4096, 11008, 512, 32, "swiglu", "bf16")]


@pytest.mark.parametrize("d,f,h,G,act,dt", CC_SHAPES)
@pytest.mark.parametrize("B", [2, 3, 4])
def test_cuda_core_arm_matches_oracle(sffn, d, f, h, G, act, dt, B):
    spec = W.LayerSpec(name="t", d=d, f=f, h=h, group_size=G, act=act, wdtype=dt, p_mean=0.12, zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=40 + B, max_batch=32, biases=(B == 3))
    L.set_batch_path("cuda_cores")
    X = W.make_tokens(d, 1, seed=B, batch=B, device="cuda")[0]
    masks, y, xo = _run(sffn, L, X, 0.0, x_out=True)
    _check_batch(host, spec, X, 0.0, masks, y)
    assert torch.equal(xo, X + y)
    L.check_error()


def test_cuda_core_arm_forward_and_predict_views(sffn):
    """Caller masks through sffn_forward (the union formed from them) and
    sffn_predict's views, on the CUDA-core arm; B = 5 falls to the tensor cores."""
    spec = W.LayerSpec(name="t", d=1024, f=2048, h=128, group_size=32, act="relu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=12, max_batch=32)
    L.set_batch_path("cuda_cores")
    B = 4
    rng = np.random.default_rng(13)
    bits = rng.random((B, spec.f)) < np.array([0.0, 1.0, 0.01, 0.3])[:, None]
    masks = L.masks(B)
    masks.nmask.copy_(torch.from_numpy(np.stack([O.bits_to_words(b).view(np.int32) for b in bits])).cuda())
    X = W.make_tokens(spec.d, 1, seed=14, batch=B, device="cuda")[0]
    y = torch.empty(B, spec.d, device="cuda")
    sffn.sffn_forward(L.handle, X, B, masks, y, None, L.workspace(B))
    torch.cuda.synchronize()
    for b in range(B):
        check_y(y[b].cpu().numpy(), host.ffn(X[b].double().cpu().numpy(), bits[b], "relu"), "bf16", f"y[{b}]")
    assert (y[0] == 0).all()
    union = bits.any(axis=0)
    assert masks.ucount.item() == int(union.sum())
    assert np.array_equal(words_bits(masks.unmask.cpu().numpy(), spec.f), union)
    m1 = L.masks(B)
    sffn.sffn_predict(L.handle, X, B, 0.0, m1, L.workspace(B))
    m2, y2, _ = _run(sffn, L, X, 0.0)
    for k in ("nmask", "gmask", "count", "unmask", "ugmask", "ucount"):
        assert torch.equal(getattr(m1, k), getattr(m2, k)), k
    X5 = W.make_tokens(spec.d, 1, seed=15, batch=5, device="cuda")[0]
    m5, y5, _ = _run(sffn, L, X5, 0.0)
    _check_batch(host, spec, X5, 0.0, m5, y5)
    L.check_error()


def test_cuda_core_arm_full_size_falcon(sffn):
    spec = W.WORKLOADS["falcon40b_relu_d8192_f32768_fp16_batch"]
    L, w, host = make_layer(spec, seed=0, max_batch=32)
    L.set_batch_path("cuda_cores")
    B = 4
    X = W.make_tokens(spec.d, 1, seed=0, batch=B, device="cuda")[0]
    masks, y, _ = _run(sffn, L, X, spec.thres)
    for b in range(B):
        xs = X[b].double().cpu().numpy()
        check_masks(host.scores(xs), spec.thres, spec.group_size, masks.nmask[b].cpu().numpy(),
                    masks.gmask[b].cpu().numpy(), masks.idx[b].cpu().numpy(), masks.count[b].item())
        if b in (0, B - 1):
            gb = words_bits(masks.nmask[b].cpu().numpy(), spec.f)
            check_y(y[b].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype, f"y[{b}]")
    L.check_error()
