"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every case draws seeded synthetic weights on the GPU, packs them through
sffn_layer_pack, runs the hot calls and compares with the oracle on the same
stored values: mask views bit-exact outside the +-1e-3 score band, y within
the stated tolerances (teacher-forced on the GPU's own mask), momentum state
bit-exact.
"""

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gb300 import workload as W
from oracle import sffn_oracle as O

from gpu_util import BAND, HostLayer, check_masks, check_y, make_layer, words_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn as mod
    return mod


def _decode(sffn, L, x, thres, masks=None, ws=None, x_out=False):
    masks = masks or L.masks()
    ws = ws if ws is not None else L.workspace()
    y = torch.empty(1, L.d, device="cuda")
    xo = torch.empty(1, L.d, device="cuda") if x_out else None
    sffn.sffn_decode_step(L.handle, x, 1, thres, masks, y, xo, ws)
    return masks, y, xo


def _token_check(L, host, act, wdtype, G, x, thres, masks, y):
    xs = x[0].double().cpu().numpy()
    s = host.scores(xs)
    m = check_masks(s, thres, G, masks.nmask[0].cpu().numpy(), masks.gmask[0].cpu().numpy(),
                    masks.idx[0].cpu().numpy(), masks.count[0].item())
    gb = words_bits(masks.nmask[0].cpu().numpy(), host.f)
    r = check_y(y[0].cpu().numpy(), host.ffn(xs, gb, act), wdtype)
    return m, r


# ------------------------------------------------------------------ small shapes, every dtype and activation

SMALL = [
    # d, f, h, G, act, dtype  (ragged: d not a power of two, f/32 words not a multiple of anything)
    (512, 2048, 64, 32, "relu", "f32"),
    (1032, 1088, 72, 64, "reglu", "bf16"),
    (776, 960, 128, 32, "swiglu", "f16"),
    (2048, 4096, 256, 32, "relu", "f16"),
    (4096, 2048, 512, 64, "swiglu", "bf16"),
    (8192, 1024, 1024, 64, "reglu", "bf16"),
    (24, 64, 16, 32, "reglu", "f32"),
    (8, 32, 8, 32, "relu", "bf16"),
    (1536, 2048, 96, 32, "relu2", "bf16"),
    (520, 960, 64, 32, "relu2", "f32"),
]


@pytest.mark.parametrize("d,f,h,G,act,dt", SMALL)
def test_decode_step_small_shapes(sffn, d, f, h, G, act, dt):
    spec = W.LayerSpec(name="t", d=d, f=f, h=h, group_size=G, act=act, wdtype=dt, p_mean=0.15,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=1, biases=(d % 3 == 0))
    X = W.make_tokens(d, 6, seed=2, device="cuda")
    for t in range(X.shape[0]):
        masks, y, _ = _decode(sffn, L, X[t], 0.0)
        _token_check(L, host, act, dt, G, X[t], 0.0, masks, y)
    L.check_error()


def test_pack_roundtrip(sffn):
    spec = W.LayerSpec(name="t", d=1032, f=1088, h=72, group_size=64, act="reglu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=3, biases=True)
    pv = L.packed()
    perm = w["perm"].long()

    def read(ptr, numel, dtype):
        return sffn.view_device(ptr, (numel,), dtype).clone()

    f, d, h = spec.f, spec.d, spec.h
    assert torch.equal(read(pv.W1, h * d, torch.bfloat16).view(h, d), w["W1"])
    assert torch.equal(read(pv.W2, f * h, torch.bfloat16).view(f, h), w["W2"][perm])
    assert torch.equal(read(pv.up, f * d, torch.bfloat16).view(f, d), w["up"][perm])
    assert torch.equal(read(pv.gate, f * d, torch.bfloat16).view(f, d), w["gate"][perm])
    assert torch.equal(read(pv.downT, f * d, torch.bfloat16).view(f, d), w["down"].t()[perm])
    assert torch.equal(read(pv.b2, f, torch.float32), w["b2"][perm])
    assert torch.equal(read(pv.b1, h, torch.float32), w["b1"])
    assert torch.equal(read(pv.perm, f, torch.int32), w["perm"])


def test_pack_rejects_non_permutation(sffn):
    spec = W.LayerSpec(name="t", d=64, f=128, h=16, group_size=32, act="relu", wdtype="f16", p_mean=0.1,
                       zipf_alpha=1.0)
    w = W.make_layer(spec, seed=0, device="cuda")
    L = sffn.Layer(spec.d, spec.f, spec.h, 32, "relu", "f16")
    bad = w["perm"].clone()
    bad[5] = bad[6]
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_layer_pack(L.handle, w["W1"], None, w["W2"], None, w["up"], None, w["down"], bad)
    assert e.value.status == sffn.SFFN_ERR_DEVICE
    bad[5] = spec.f  # out of range
    with pytest.raises(sffn.SffnError):
        sffn.sffn_layer_pack(L.handle, w["W1"], None, w["W2"], None, w["up"], None, w["down"], bad)
    L.check_error()


# ------------------------------------------------------------------ special cases

@pytest.mark.parametrize("act,dt", [("relu", "f32"), ("reglu", "bf16"), ("swiglu", "f16"), ("relu2", "bf16")])
def test_all_active_and_none_active(sffn, act, dt):
    spec = W.LayerSpec(name="t", d=1024, f=2048, h=128, group_size=32, act=act, wdtype=dt, p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=4)
    x = W.make_tokens(spec.d, 1, seed=5, device="cuda")[0]
    masks, y, xo = _decode(sffn, L, x, float("-inf"), x_out=True)
    assert masks.count.item() == spec.f
    assert (masks.nmask == -1).all()
    xs = x[0].double().cpu().numpy()
    # all active: the oracle's dense FFN on the same stored weights
    U = O.widen(host.up, dt)
    G = O.widen(host.gate, dt) if host.gate is not None else None
    Dn = O.widen(host.down, dt)
    check_y(y[0].cpu().numpy(), O.ffn_dense(xs, U, G, Dn, act), dt)
    assert torch.allclose(xo, x + y, rtol=0, atol=0)
    masks, y, xo = _decode(sffn, L, x, float("inf"), x_out=True)
    assert masks.count.item() == 0 and (masks.nmask == 0).all() and (masks.gmask == 0).all()
    assert (y == 0).all()
    assert torch.equal(xo, x)
    L.check_error()


def test_nan_input_marks_nothing_active(sffn):
    spec = W.LayerSpec(name="t", d=256, f=512, h=64, group_size=32, act="relu", wdtype="f16", p_mean=0.2,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=6)
    x = torch.full((1, spec.d), float("nan"), device="cuda")
    masks, y, _ = _decode(sffn, L, x, 0.0)
    assert masks.count.item() == 0 and (y == 0).all()


def test_caller_masks_forward(sffn):
    spec = W.LayerSpec(name="t", d=2048, f=4096, h=128, group_size=64, act="reglu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=7)
    rng = np.random.default_rng(0)
    ws = L.workspace()
    for trial in range(6):
        frac = [0.0, 1.0, 0.01, 0.3, 0.7, 1.0 / spec.f][trial]
        bits = rng.random(spec.f) < frac
        if trial == 5:
            bits[:] = False
            bits[spec.f - 1] = True           # one neuron, the last slot
        words = O.bits_to_words(bits).view(np.int32)
        masks = L.masks()
        masks.nmask[0] = torch.from_numpy(words).cuda()
        x = W.make_tokens(spec.d, 1, seed=10 + trial, device="cuda")[0]
        y = torch.empty(1, spec.d, device="cuda")
        sffn.sffn_forward(L.handle, x, 1, masks, y, None, ws)
        check_y(y[0].cpu().numpy(), host.ffn(x[0].double().cpu().numpy(), bits, "reglu"), "bf16")
    L.check_error()


def test_predict_views_match_decode(sffn):
    spec = W.WORKLOADS["relu_d512_f2048_fp32"]
    L, w, host = make_layer(spec, seed=0)
    x = W.make_tokens(spec.d, 1, seed=1, device="cuda")[0]
    m1 = L.masks()
    sffn.sffn_predict(L.handle, x, 1, 0.0, m1, L.workspace())
    m2, y, _ = _decode(sffn, L, x, 0.0)
    for k in ("nmask", "gmask", "count"):
        assert torch.equal(getattr(m1, k), getattr(m2, k))
    c = m1.count.item()
    assert torch.equal(m1.idx[0, :c], m2.idx[0, :c])


def test_deterministic(sffn):
    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"], f=4096, tam_capacity=None)
    L, w, host = make_layer(spec, seed=8)
    x = W.make_tokens(spec.d, 1, seed=9, device="cuda")[0]
    _, y1, _ = _decode(sffn, L, x, 0.0)
    _, y2, _ = _decode(sffn, L, x, 0.0)
    assert torch.equal(y1, y2)


def test_l2_hint_leaves_results_unchanged(sffn):
    """sffn_layer_set_next only warms L2: masks, y and x + y are bit-identical
    with the hint on (to another layer, to the layer itself) and off."""
    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"], f=4096, tam_capacity=None)
    A, _, _ = make_layer(spec, seed=0, layer=0)
    Bl, _, _ = make_layer(spec, seed=0, layer=1)
    x = W.make_tokens(spec.d, 1, seed=2, kind="ar1", device="cuda")[0]
    m0, y0, xo0 = _decode(sffn, A, x, 0.0, x_out=True)
    for nxt in (Bl, A, None):
        A.set_next(nxt)
        m1, y1, xo1 = _decode(sffn, A, x, 0.0, x_out=True)
        assert torch.equal(y0, y1) and torch.equal(xo0, xo1)
        for k in ("nmask", "gmask", "idx", "count"):
            assert torch.equal(getattr(m0, k), getattr(m1, k)), k
    # hot groups read with the L2 keep priority: also unchanged
    n_gw = (spec.f // spec.group_size + 31) // 32
    res = torch.randint(0, 2**31, (n_gw,), dtype=torch.int32, device="cuda")
    A.set_l2_resident(res)
    m1, y1, xo1 = _decode(sffn, A, x, 0.0, x_out=True)
    assert torch.equal(y0, y1) and torch.equal(xo0, xo1) and torch.equal(m0.idx, m1.idx)
    A.set_l2_resident(None)
    A.set_next(Bl)
    y2 = torch.empty(1, spec.d, device="cuda")
    m2 = A.masks()
    sffn.sffn_decode_step_static_ws(A.handle, x, 1, 0.0, m2, y2, None)
    assert torch.equal(y0, y2)
    A.check_error()


# ------------------------------------------------------------------ tiny workload: 64 tokens with momentum

def test_tiny_sequence_with_tam(sffn):
    spec = W.WORKLOADS["relu_d512_f2048_fp32"]
    L, w, host = make_layer(spec, seed=0)
    tam = sffn.Tam(1, spec.n_groups, spec.tam_lambda)
    outs = sffn.TamOutputs(1, spec.n_groups, spec.capacity)
    X = W.make_tokens(spec.d, spec.tokens, seed=0, kind=spec.seq, device="cuda")
    s_ref = np.zeros(spec.n_groups, dtype=np.float32)
    prev = np.zeros(spec.n_groups, dtype=bool)
    masks, ws = L.masks(), L.workspace()
    y = torch.empty(1, spec.d, device="cuda")
    scores_dev = torch.empty(spec.n_groups, device="cuda")
    band_total = 0
    for t in range(spec.tokens):
        sffn.sffn_decode_step(L.handle, X[t], 1, spec.thres, masks, y, None, ws)
        sffn.tam_update(tam.handle, 0, 1, masks.gmask, masks.gwords, -1.0, spec.tam_eps, spec.capacity, outs)
        m, _ = _token_check(L, host, spec.act, spec.wdtype, spec.group_size, X[t], spec.thres, masks, y)
        band_total += m["band"]
        ga = words_bits(masks.gmask[0].cpu().numpy(), spec.n_groups)
        r = O.tam_update(s_ref, prev, ga, np.float32(spec.tam_lambda), np.float32(spec.tam_eps), spec.capacity)
        s_ref, prev = r["scores"], r["resident"]
        sffn.tam_get_state(tam.handle, scores_dev, None, None)
        assert np.array_equal(scores_dev.cpu().numpy(), s_ref), t   # bit-exact float32
        n = spec.n_groups
        assert np.array_equal(words_bits(outs.cand[0].cpu().numpy(), n), r["cand"])
        assert np.array_equal(words_bits(outs.resident[0].cpu().numpy(), n), r["resident"])
        assert np.array_equal(words_bits(outs.load[0].cpu().numpy(), n), r["load"])
        assert np.array_equal(words_bits(outs.evict[0].cpu().numpy(), n), r["evict"])
        assert np.array_equal(words_bits(outs.changed[0].cpu().numpy(), n), r["changed"])
        k = r["topk"].shape[0]
        assert outs.n_cand[0].item() == r["n_cand"] and outs.n_res[0].item() == k
        assert np.array_equal(outs.topk[0, :k].cpu().numpy(), r["topk"])
        assert (outs.topk[0, k:] == -1).all()
    assert band_total < 2 * spec.tokens
    L.check_error()
    sffn.tam_check_error(tam.handle)


def test_tam_scripted_and_adapt(sffn):
    """Momentum on scripted group sequences (closed forms of the oracle pins),
    many layers at once, lambda override, state round trip and the lambda step."""
    n_layers, n_groups = 5, 1000
    tam = sffn.Tam(n_layers, n_groups, 0.9)
    gw = (n_groups + 31) // 32
    rng = np.random.default_rng(1)
    lam_l = np.full(n_layers, 0.9, dtype=np.float32)
    s_ref = np.zeros((n_layers, n_groups), dtype=np.float32)
    prev = np.zeros((n_layers, n_groups), dtype=bool)
    K = 300
    outs = sffn.TamOutputs(n_layers, n_groups, K)
    stall_all = W.make_stall_bits(40, n_layers, seed=3)
    for t in range(40):
        A = rng.random((n_layers, n_groups)) < rng.random()
        gm = np.stack([O.bits_to_words(A[l]) for l in range(n_layers)]).view(np.int32)
        gm_dev = torch.from_numpy(np.ascontiguousarray(gm)).cuda()
        lam_arg = 0.95 if t % 7 == 3 else -1.0
        sffn.tam_update(tam.handle, 0, n_layers, gm_dev, gw, lam_arg, 0.01, K, outs)
        for l in range(n_layers):
            lam = np.float32(lam_arg) if lam_arg >= 0 else lam_l[l]
            r = O.tam_update(s_ref[l], prev[l], A[l], lam, np.float32(0.01), K)
            s_ref[l], prev[l] = r["scores"], r["resident"]
            kk = r["topk"].shape[0]
            assert np.array_equal(outs.topk[l, :kk].cpu().numpy(), r["topk"]), (t, l)
            assert np.array_equal(words_bits(outs.load[l].cpu().numpy(), n_groups), r["load"])
        stall = torch.from_numpy(stall_all[t]).cuda()
        sffn.tam_adapt(tam.handle, 0, n_layers, stall, 0.01, 0.8, 0.99)
        for l in range(n_layers):
            lam_l[l] = O.anb_step(lam_l[l], bool(stall_all[t, l]), 0.01, 0.8, 0.99)
    sc = torch.empty(n_layers, n_groups, device="cuda")
    la = torch.empty(n_layers, device="cuda")
    rs = torch.empty(n_layers, gw, dtype=torch.int32, device="cuda")
    sffn.tam_get_state(tam.handle, sc, la, rs)
    assert np.array_equal(sc.cpu().numpy(), s_ref)
    assert np.array_equal(la.cpu().numpy(), lam_l)
    # checkpoint / resume into a fresh state gives identical next steps
    tam2 = sffn.Tam(n_layers, n_groups, 0.5)
    sffn.tam_set_state(tam2.handle, sc, la, rs)
    gm_dev = torch.from_numpy(np.stack([O.bits_to_words(rng.random(n_groups) < 0.3)
                                        for _ in range(n_layers)]).view(np.int32)).cuda()
    o1, o2 = sffn.TamOutputs(n_layers, n_groups, K), sffn.TamOutputs(n_layers, n_groups, K)
    sffn.tam_update(tam.handle, 0, n_layers, gm_dev, gw, -1.0, 0.01, K, o1)
    sffn.tam_update(tam2.handle, 0, n_layers, gm_dev, gw, -1.0, 0.01, K, o2)
    assert torch.equal(o1.topk, o2.topk) and torch.equal(o1.resident, o2.resident)
    # scripted: isolated hit never a candidate; hit after m misses rule
    t3 = sffn.Tam(1, 32, 0.9)
    o3 = sffn.TamOutputs(1, 32, 32)
    one = torch.tensor([[1]], dtype=torch.int32, device="cuda")
    zero = torch.tensor([[0]], dtype=torch.int32, device="cuda")
    sffn.tam_update(t3.handle, 0, 1, one, 1, -1.0, 0.01, 32, o3)
    assert o3.n_cand.item() == 0
    for _ in range(20):
        sffn.tam_update(t3.handle, 0, 1, zero, 1, -1.0, 0.01, 32, o3)
    sffn.tam_update(t3.handle, 0, 1, one, 1, -1.0, 0.01, 32, o3)
    assert o3.n_cand.item() == 1 and o3.topk[0, 0].item() == 0
    sffn.tam_check_error(tam.handle)


# ------------------------------------------------------------------ full-size layers, a few tokens

FULL = [
    ("opt6.7b_relu_d4096_f16384_fp16", 3),
    ("llama2_70b_reglu_d8192_f28672_bf16_8l", 2),
    ("falcon40b_relu_d8192_f32768_fp16_batch", 2),
    ("swiglu7b_d4096_f11008_bf16_32l", 2),
]


@pytest.mark.parametrize("name,T", FULL)
def test_full_size_layer(sffn, name, T):
    spec = W.WORKLOADS[name]
    L, w, host = make_layer(spec, seed=0)
    X = W.make_tokens(spec.d, T, seed=0, kind=spec.seq, device="cuda")
    for t in range(T):
        masks, y, _ = _decode(sffn, L, X[t], spec.thres)
        m, r = _token_check(L, host, spec.act, spec.wdtype, spec.group_size, X[t], spec.thres, masks, y)
        frac = m["active"] / spec.f
        assert abs(frac - spec.p_mean) < 0.5 * spec.p_mean
    L.check_error()


def test_stack_residual_teacher_forced(sffn):
    """Two layers of the 70B-shaped stack: x_{l+1} = x_l + y_l; each layer is
    checked against the oracle on the GPU's own input (teacher forcing)."""
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"]
    layers = [make_layer(spec, seed=0, layer=l) for l in range(2)]
    x = W.make_tokens(spec.d, 1, seed=4, kind="ar1", device="cuda")[0]
    for l, (L, w, host) in enumerate(layers):
        masks, y, xo = _decode(sffn, L, x, spec.thres, x_out=True)
        _token_check(L, host, spec.act, spec.wdtype, spec.group_size, x, spec.thres, masks, y)
        assert torch.equal(xo, x + y)
        x = xo


def test_timeout_path_reports_and_recovers(sffn):
    spec = W.LayerSpec(name="t", d=64, f=64, h=8, group_size=32, act="relu", wdtype="f16", p_mean=0.2,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=0)
    sffn.sffn_selftest_wait_timeout(L.handle, 2000)
    with pytest.raises(sffn.SffnError) as e:
        L.check_error()
    assert e.value.status == sffn.SFFN_ERR_TIMEOUT
    L.check_error()          # cleared
    x = W.make_tokens(spec.d, 1, seed=0, device="cuda")[0]
    masks, y, _ = _decode(sffn, L, x, 0.0)   # the context is still usable
    _token_check(L, host, "relu", "f16", 32, x, 0.0, masks, y)


def test_batch_above_one_needs_16bit_weights(sffn):
    spec = W.LayerSpec(name="t", d=64, f=64, h=8, group_size=32, act="relu", wdtype="f32", p_mean=0.2,
                       zipf_alpha=1.0)
    w = W.make_layer(spec, seed=0, device="cuda")
    L = sffn.Layer.from_weights(w, 32, "relu", max_batch=4)
    x = torch.zeros(4, 64, device="cuda")
    y = torch.empty(4, 64, device="cuda")
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_decode_step(L.handle, x, 4, 0.0, L.masks(4), y, None, L.workspace(1))
    assert e.value.status == sffn.SFFN_ERR_UNSUPPORTED
