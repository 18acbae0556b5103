"""Parity cases for launch shapes and sequence lengths the other GPU tests do
not reach, through the C ABI against the oracle:

* fp32 layers whose rows are longer than 16 KB (d = 6144 and 8192): the FFN
  and predictor kernels' eight-chunks-per-thread instantiations;
* finite, non-zero thresholds at B = 1 and on the batched (B >= 16) path;
* every layer of the 8-layer 70B-shaped stack, teacher-forced, with the L2
  hint linking each layer to the next as the bench runs it;
* the momentum state over the 70B stack's full 512-token sequence and over
  the 32-layer SwiGLU loop's 1024 tokens with the topic shift at token 512
  and the adaptive lambda step, bit-exact every token, fed by the GPU's own
  group masks; the composite per-layer call (predict, FFN, momentum) and the
  batched all-layer momentum call must agree;
* the L2 residency hint driven by a momentum state's resident set, checked
  against the oracle.
"""

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gb300 import workload as W
from oracle import sffn_oracle as O

from gpu_util import HostLayer, check_masks, check_y, make_layer, words_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn as mod
    return mod


def _decode(sffn, L, x, thres, x_out=False):
    masks, ws = L.masks(), L.workspace()
    y = torch.full((1, L.d), float("nan"), device="cuda")
    xo = torch.empty(1, L.d, device="cuda") if x_out else None
    sffn.sffn_decode_step(L.handle, x, 1, thres, masks, y, xo, ws)
    torch.cuda.synchronize()
    return masks, y, xo


def _check_token(host, spec, x, thres, masks, y, b=0):
    xs = x.double().cpu().numpy().reshape(-1)
    s = host.scores(xs)
    m = check_masks(s, thres, spec.group_size, masks.nmask[b].cpu().numpy(), masks.gmask[b].cpu().numpy(),
                    masks.idx[b].cpu().numpy(), masks.count[b].item())
    gb = words_bits(masks.nmask[b].cpu().numpy(), spec.f)
    check_y(y[b].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype)
    return m


# ------------------------------------------------------------------ fp32 rows above 16 KB

@pytest.mark.parametrize("d,act", [(6144, "relu"), (6144, "reglu"), (8192, "swiglu"), (8192, "relu2")])
def test_fp32_long_rows(sffn, d, act):
    spec = W.LayerSpec(name="t", d=d, f=2048, h=256, group_size=32, act=act, wdtype="f32", p_mean=0.12,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=21, biases=True)
    X = W.make_tokens(d, 3, seed=22, device="cuda")
    for t in range(X.shape[0]):
        masks, y, _ = _decode(sffn, L, X[t], 0.0)
        m = _check_token(host, spec, X[t], 0.0, masks, y)
        assert 0 < m["active"] < spec.f
    L.check_error()


# ------------------------------------------------------------------ finite thresholds

@pytest.mark.parametrize("thres", [-0.05, 0.1])
def test_finite_threshold_single_token(sffn, thres):
    spec = W.LayerSpec(name="t", d=2048, f=4096, h=256, group_size=64, act="reglu", wdtype="bf16", p_mean=0.15,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=23, biases=True)
    X = W.make_tokens(spec.d, 4, seed=24, device="cuda")
    counts = []
    for t in range(X.shape[0]):
        masks, y, _ = _decode(sffn, L, X[t], thres)
        counts.append(_check_token(host, spec, X[t], thres, masks, y)["active"])
        # the threshold matters: at 0 the active set differs
        m0, _, _ = _decode(sffn, L, X[t], 0.0)
        assert not torch.equal(m0.nmask, masks.nmask)
    assert min(counts) > 0
    L.check_error()


@pytest.mark.parametrize("thres", [-0.05, 0.1])
@pytest.mark.parametrize("B", [16, 32])
def test_finite_threshold_batch(sffn, thres, B):
    spec = W.LayerSpec(name="t", d=1024, f=4096, h=128, group_size=64, act="reglu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=25, max_batch=32, biases=True)
    X = W.make_tokens(spec.d, 1, seed=26, batch=B, device="cuda")[0]
    masks, ws = L.masks(B), L.workspace(B)
    y = torch.full((B, spec.d), float("nan"), device="cuda")
    sffn.sffn_decode_step(L.handle, X, B, thres, masks, y, None, ws)
    torch.cuda.synchronize()
    union = np.zeros(spec.f, dtype=bool)
    for b in range(B):
        _check_token(host, spec, X[b], thres, masks, y, b)
        union |= words_bits(masks.nmask[b].cpu().numpy(), spec.f)
    assert np.array_equal(words_bits(masks.unmask.cpu().numpy(), spec.f), union)
    assert masks.ucount.item() == int(union.sum())
    L.check_error()


# ------------------------------------------------------------------ the 8-layer 70B-shaped stack

def _stack(sffn, spec, seed=0):
    layers = []
    for l in range(spec.layers):
        w = W.make_layer(spec, seed=seed, layer=l, device="cuda")
        layers.append(sffn.Layer.from_weights(w, spec.group_size, spec.act))
        del w
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return layers


def test_70b_stack_every_layer_teacher_forced(sffn):
    """Two tokens through all eight layers with x_{l+1} = x_l + y_l and the
    next-layer L2 hint on (as the bench runs the stack); each layer's masks and
    y against the oracle on the GPU's own layer input."""
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"]
    nL, T = spec.layers, 2
    layers = _stack(sffn, spec)
    for l in range(nL):
        layers[l].set_next(layers[(l + 1) % nL])
    X = W.spec_tokens(spec, T, seed=0, device="cuda")[:, 0]
    ws = layers[0].workspace()
    saved = {}
    for t in range(T):
        x = X[t:t + 1].contiguous()
        for l, L in enumerate(layers):
            masks = L.masks()
            y = torch.empty(1, spec.d, device="cuda")
            xo = torch.empty(1, spec.d, device="cuda")
            sffn.sffn_decode_step(L.handle, x, 1, spec.thres, masks, y, xo, ws)
            torch.cuda.synchronize()
            assert torch.equal(xo, x + y)
            saved[(t, l)] = (x.clone(), masks, y.clone())
            x = xo
    for l in range(nL):
        w = W.make_layer(spec, seed=0, layer=l, device="cuda")
        host = HostLayer(w, spec.wdtype)
        del w
        for t in range(T):
            x, masks, y = saved[(t, l)]
            m = _check_token(host, spec, x[0], spec.thres, masks, y)
            assert abs(m["active"] / spec.f - spec.p_mean) < 0.5 * spec.p_mean, (t, l)
        del host
    for L in layers:
        L.check_error()


# ------------------------------------------------------------------ momentum over whole sequences

def _tam_rows(sffn, n_layers, n_groups, K):
    """One single-layer output set per layer (the composite call writes row 0 of its outputs)."""
    return [sffn.TamOutputs(1, n_groups, K) for _ in range(n_layers)]


def _check_tam_token(r_layers, outs_rows, n_groups, t):
    for l, r in enumerate(r_layers):
        o = outs_rows[l]
        k = r["topk"].shape[0]
        assert o["n_cand"] == r["n_cand"] and o["n_res"] == k, (t, l)
        assert np.array_equal(o["topk"][:k], r["topk"]), (t, l)
        assert (o["topk"][k:] == -1).all(), (t, l)
        for key in ("cand", "resident", "load", "evict", "changed"):
            assert np.array_equal(words_bits(o[key], n_groups), r[key]), (t, l, key)


def test_tam_over_70b_stack_512_tokens(sffn):
    """The 70B-shaped stack's full 512-token sequence: every layer through
    sffn_decode_step_tam (predict, FFN, then that layer's momentum step on the
    group mask it wrote). The momentum scores and output sets equal the
    oracle's float32 recursion fed the GPU's group masks, bit for bit, every
    token; a second state updated by one batched tam_update over all layers
    per token ends identical; each group mask is the OR of its neuron words."""
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"]
    nL, ng, G, f = spec.layers, spec.n_groups, spec.group_size, spec.f
    T, K = spec.tokens, spec.capacity
    layers = _stack(sffn, spec)
    for l in range(nL):
        layers[l].set_next(layers[(l + 1) % nL])
    gw = (ng + 31) // 32
    tam = sffn.Tam(nL, ng, spec.tam_lambda)
    tam_b = sffn.Tam(nL, ng, spec.tam_lambda)
    rows = _tam_rows(sffn, nL, ng, K)
    outs_b = sffn.TamOutputs(nL, ng, K)
    X = W.spec_tokens(spec, T, seed=0, device="cuda")[:, 0]
    masks = [L.masks() for L in layers]
    ws = layers[0].workspace()
    y = torch.empty(1, spec.d, device="cuda")
    xa, xb = torch.empty(1, spec.d, device="cuda"), torch.empty(1, spec.d, device="cuda")
    gm_all = torch.zeros(nL, gw, dtype=torch.int32, device="cuda")
    s_ref = np.zeros((nL, ng), dtype=np.float32)
    prev = np.zeros((nL, ng), dtype=bool)
    lam, eps = np.float32(spec.tam_lambda), np.float32(spec.tam_eps)
    sc = torch.empty(nL, ng, device="cuda")
    nonzero_load = 0
    for t in range(T):
        x = X[t:t + 1]
        for l in range(nL):
            xo = (xa, xb)[l % 2]
            sffn.sffn_decode_step_tam(layers[l].handle, tam.handle, l, x, 1, spec.thres, masks[l], y, xo, ws,
                                      -1.0, spec.tam_eps, K, rows[l])
            gm_all[l].copy_(masks[l].gmask[0])
            x = xo
        sffn.tam_update(tam_b.handle, 0, nL, gm_all, gw, -1.0, spec.tam_eps, K, outs_b)
        sffn.tam_get_state(tam.handle, sc, None, None)
        host = [{k: getattr(o, k)[0].cpu().numpy() for k in ("cand", "resident", "load", "evict", "changed", "topk")}
                | {"n_cand": o.n_cand.item(), "n_res": o.n_res.item()} for o in rows]
        nw = torch.stack([m.nmask[0] for m in masks]).cpu().numpy()
        gms = gm_all.cpu().numpy()
        r_layers = []
        for l in range(nL):
            nb = words_bits(nw[l], f)
            ga = words_bits(gms[l], ng)
            assert np.array_equal(ga, nb.reshape(ng, G).any(axis=1)), (t, l)
            r = O.tam_update(s_ref[l], prev[l], ga, lam, eps, K)
            s_ref[l], prev[l] = r["scores"], r["resident"]
            r_layers.append(r)
            nonzero_load += int(r["load"].any())
        _check_tam_token(r_layers, host, ng, t)
        assert np.array_equal(sc.cpu().numpy(), s_ref), t
    # the two schedules of the momentum step leave identical states and outputs
    sb = torch.empty(nL, ng, device="cuda")
    rb = torch.empty(nL, gw, dtype=torch.int32, device="cuda")
    ra = torch.empty(nL, gw, dtype=torch.int32, device="cuda")
    sffn.tam_get_state(tam_b.handle, sb, None, rb)
    sffn.tam_get_state(tam.handle, sc, None, ra)
    assert torch.equal(sb, sc) and torch.equal(ra, rb)
    assert nonzero_load > nL      # the resident sets move along the sequence
    for L in layers:
        L.check_error()
    sffn.tam_check_error(tam.handle)


def test_swiglu_loop_1024_tokens_topic_shift(sffn):
    """The 32-layer SwiGLU loop over its full 1024 tokens with the group ranks
    redrawn at token 512 and the adaptive lambda step after every token: the
    momentum state and lambdas bit-exact against the oracle every token (fed
    the GPU's group masks); masks and y against the oracle on the first and
    last layer at the tokens either side of the shift and at the ends. Each
    layer is fed x_l / rms(x_l) (harness stand-in for the block's
    normalisation; the FFN path is unchanged)."""
    spec = W.WORKLOADS["swiglu7b_d4096_f11008_bf16_32l"]
    nL, ng, G, f = spec.layers, spec.n_groups, spec.group_size, spec.f
    T, shift, K = spec.tokens, spec.topic_shift_at, spec.capacity
    gw = (ng + 31) // 32
    layers = []
    for l in range(nL):
        w = W.make_layer(spec, seed=0, layer=l, device="cuda")
        layers.append(sffn.Layer.from_weights(w, G, spec.act))
        del w
    check_tok = {0, shift - 1, shift, T - 1}
    check_layers = (0, nL - 1)
    tam = sffn.Tam(nL, ng, spec.tam_lambda)
    outs = sffn.TamOutputs(nL, ng, K)
    stalls = W.make_stall_bits(T, nL, seed=0)
    stalls_dev = torch.from_numpy(stalls).cuda()
    s_ref = np.zeros((nL, ng), dtype=np.float32)
    prev = np.zeros((nL, ng), dtype=bool)
    lam = np.full(nL, spec.tam_lambda, dtype=np.float32)
    eps = np.float32(spec.tam_eps)
    X = W.spec_tokens(spec, T, seed=0, device="cuda")[:, 0]
    masks = [L.masks() for L in layers]
    ws = layers[0].workspace()
    y = torch.empty(1, spec.d, device="cuda")
    xo = torch.empty(1, spec.d, device="cuda")
    gm_all = torch.zeros(nL, gw, dtype=torch.int32, device="cuda")
    sc = torch.empty(nL, ng, device="cuda")
    la = torch.empty(nL, device="cuda")
    saved = {}
    frac = []
    for t in range(T):
        if t == shift:
            for l in range(nL):
                w = W.make_layer(spec, seed=0, layer=l, device="cuda")
                w["W2"] = W.make_w2_topic(spec, 0, l, 1, w["W1"], w["perm"])
                layers[l].pack(w)
                del w
            torch.cuda.synchronize()
        resid = X[t:t + 1].clone()
        for l in range(nL):
            x = resid / torch.sqrt((resid * resid).mean())
            sffn.sffn_decode_step(layers[l].handle, x, 1, spec.thres, masks[l], y, xo, ws)
            gm_all[l].copy_(masks[l].gmask[0])
            if t in check_tok and l in check_layers:
                saved[(t, l)] = (x.clone(), torch.stack([masks[l].nmask[0]]).clone(), masks[l].gmask.clone(),
                                 masks[l].idx.clone(), masks[l].count.clone(), y.clone())
            resid = resid + y
        sffn.tam_update(tam.handle, 0, nL, gm_all, gw, -1.0, spec.tam_eps, K, outs)
        sffn.tam_adapt(tam.handle, 0, nL, stalls_dev[t], spec.anb_alpha, spec.anb_lo, spec.anb_hi)
        sffn.tam_get_state(tam.handle, sc, la, None)
        gms = gm_all.cpu().numpy()
        topk = outs.topk.cpu().numpy()
        res = outs.resident.cpu().numpy()
        chg = outs.changed.cpu().numpy()
        ncand = outs.n_cand.cpu().numpy()
        frac.append(float(torch.stack([m.count[0] for m in masks]).float().mean().item()) / f)
        for l in range(nL):
            r = O.tam_update(s_ref[l], prev[l], words_bits(gms[l], ng), lam[l], eps, K)
            s_ref[l], prev[l] = r["scores"], r["resident"]
            k = r["topk"].shape[0]
            assert ncand[l] == r["n_cand"], (t, l)
            assert np.array_equal(topk[l, :k], r["topk"]), (t, l)
            assert np.array_equal(words_bits(res[l], ng), r["resident"]), (t, l)
            assert np.array_equal(words_bits(chg[l], ng), r["changed"]), (t, l)
            lam[l] = O.anb_step(lam[l], bool(stalls[t, l]), spec.anb_alpha, spec.anb_lo, spec.anb_hi)
        assert np.array_equal(sc.cpu().numpy(), s_ref), t
        assert np.array_equal(la.cpu().numpy(), lam), t
    assert abs(np.mean(frac) - spec.p_mean) < 0.1
    # lambdas move inside their clamp
    assert lam.min() >= spec.anb_lo and lam.max() <= spec.anb_hi and len(set(lam.tolist())) > 1
    # oracle checks of the saved layer-tokens (the topic-1 W2 for tokens after the shift)
    for l in check_layers:
        w0 = W.make_layer(spec, seed=0, layer=l, device="cuda")
        host0 = HostLayer(w0, spec.wdtype)
        w1 = dict(w0)
        w1["W2"] = W.make_w2_topic(spec, 0, l, 1, w0["W1"], w0["perm"])
        host1 = HostLayer(w1, spec.wdtype)
        for t in sorted(check_tok):
            x, nm, gm, idx, cnt, yy = saved[(t, l)]
            host = host1 if t >= shift else host0
            xs = x[0].double().cpu().numpy()
            s = host.scores(xs)
            check_masks(s, spec.thres, G, nm[0].cpu().numpy(), gm[0].cpu().numpy(), idx[0].cpu().numpy(),
                        cnt[0].item())
            gb = words_bits(nm[0].cpu().numpy(), f)
            check_y(yy[0].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype, f"y[t={t}, l={l}]")
        del w0, w1, host0, host1
    for L in layers:
        L.check_error()
    sffn.tam_check_error(tam.handle)


# ------------------------------------------------------------------ L2 residency from the momentum state

def test_l2_resident_from_momentum_matches_oracle(sffn):
    """The hot-group hint as the bench drives it: a momentum state whose
    capacity is a few groups picks each layer's resident set from the previous
    token's group masks; the FFN reads those groups' rows with the L2 keep
    priority. Masks and y of every layer-token against the oracle."""
    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"], f=8192, layers=2,
                          tam_capacity=None)
    nL, ng, T, Kl2 = spec.layers, spec.n_groups, 5, 4
    built = [make_layer(spec, seed=0, layer=l) for l in range(nL)]
    gw = (ng + 31) // 32
    tam_l2 = sffn.Tam(nL, ng, spec.tam_lambda)
    outs = sffn.TamOutputs(nL, ng, Kl2)
    for l, (L, _, _) in enumerate(built):
        L.set_l2_resident(outs.resident[l])
        L.set_next(built[(l + 1) % nL][0])
    X = W.spec_tokens(spec, T, seed=1, device="cuda")[:, 0]
    gm_all = torch.zeros(nL, gw, dtype=torch.int32, device="cuda")
    kept_any = 0
    for t in range(T):
        x = X[t:t + 1].contiguous()
        for l, (L, w, host) in enumerate(built):
            masks, y, xo = _decode(sffn, L, x, spec.thres, x_out=True)
            _check_token(host, spec, x[0], spec.thres, masks, y)
            gm_all[l].copy_(masks.gmask[0])
            x = xo
        # the next token reads the groups this token's momentum keeps
        sffn.tam_update(tam_l2.handle, 0, nL, gm_all, gw, -1.0, spec.tam_eps, Kl2, outs)
        kept_any += int(outs.n_res.sum().item())
    assert kept_any > 0
    for L, _, _ in built:
        L.set_l2_resident(None)
        L.check_error()


# ------------------------------------------------------------------ the largest layers the library accepts

def test_maximum_row_length_and_group_count(sffn):
    """d = 16384 with 16-bit weights (32 KB rows, the longest accepted) at B = 1;
    f = 65536 in 1024 groups of 64 (the most groups, 2048 mask words: the
    longest scan) at B = 1 and through the tensor-core batch path at B = 32;
    and a momentum step over all 1024 groups. Masks and y against the oracle."""
    spec = W.LayerSpec(name="t", d=16384, f=2048, h=256, group_size=32, act="relu", wdtype="bf16", p_mean=0.15,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=51)
    X = W.make_tokens(spec.d, 2, seed=52, device="cuda")
    for t in range(X.shape[0]):
        masks, y, _ = _decode(sffn, L, X[t], 0.0)
        _check_token(host, spec, X[t], 0.0, masks, y)
    L.check_error()
    del L, w, host

    spec = W.LayerSpec(name="t", d=1024, f=65536, h=128, group_size=64, act="reglu", wdtype="f16", p_mean=0.05,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=53, max_batch=32)
    X = W.make_tokens(spec.d, 2, seed=54, device="cuda")
    for t in range(X.shape[0]):
        masks, y, _ = _decode(sffn, L, X[t], 0.0)
        _check_token(host, spec, X[t], 0.0, masks, y)
    B = 32
    XB = W.make_tokens(spec.d, 1, seed=55, batch=B, device="cuda")[0]
    mb, wsb = L.masks(B), L.workspace(B)
    yb = torch.full((B, spec.d), float("nan"), device="cuda")
    sffn.sffn_decode_step(L.handle, XB, B, 0.0, mb, yb, None, wsb)
    torch.cuda.synchronize()
    union = np.zeros(spec.f, dtype=bool)
    for b in range(B):
        xs = XB[b].double().cpu().numpy()
        check_masks(host.scores(xs), 0.0, spec.group_size, mb.nmask[b].cpu().numpy(), mb.gmask[b].cpu().numpy(),
                    mb.idx[b].cpu().numpy(), mb.count[b].item())
        gb = words_bits(mb.nmask[b].cpu().numpy(), spec.f)
        union |= gb
        if b in (0, B - 1):
            check_y(yb[b].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype, f"y[{b}]")
    assert mb.ucount.item() == int(union.sum())
    # the momentum step over all 1024 groups, fed the union group mask
    ng = spec.n_groups
    tam = sffn.Tam(1, ng, 0.9)
    outs = sffn.TamOutputs(1, ng, 512)
    s_ref, prev = np.zeros(ng, dtype=np.float32), np.zeros(ng, dtype=bool)
    for _ in range(3):
        sffn.tam_update(tam.handle, 0, 1, mb.ugmask, (ng + 31) // 32, -1.0, 0.01, 512, outs)
        r = O.tam_update(s_ref, prev, words_bits(mb.ugmask.cpu().numpy(), ng), np.float32(0.9), np.float32(0.01), 512)
        s_ref, prev = r["scores"], r["resident"]
        k = r["topk"].shape[0]
        assert np.array_equal(outs.topk[0, :k].cpu().numpy(), r["topk"])
        assert np.array_equal(words_bits(outs.resident[0].cpu().numpy(), ng), r["resident"])
    L.check_error()
    sffn.tam_check_error(tam.handle)
