"""The whole-stack decode kernel (sffn_stack_decode) through the C ABI.

One launch runs every layer of a stack for one token: predictor, threshold,
sparse FFN and residual. Each case compares, layer by layer:
  * with the oracle, teacher-forced on the kernel's own layer input
    (xs[l-1]): mask views bit-exact outside the +-1e-3 score band, y within
    the tolerances of the parity tests;
  * with the per-layer chain of sffn_decode_step calls on the same input:
    the mask views, y and the residual stream are bit-identical whenever the
    masks agree (the kernel keeps the per-layer kernels' summation orders; a
    score that lands within rounding of the threshold can flip one bit, and
    then only the oracle comparison applies).
"""

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gb300 import workload as W
from oracle import sffn_oracle as O

from gpu_util import HostLayer, check_masks, check_y, words_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn as mod
    return mod


def _layers(sffn, spec, n, seed=0, biases=False):
    layers, weights = [], []
    for l in range(n):
        w = W.make_layer(spec, seed=seed, layer=l, device="cuda")
        if biases:
            g = torch.Generator(device="cuda")
            g.manual_seed(W.sub_seed(seed, "bias", l))
            w["b1"] = 0.1 * torch.randn(spec.h, generator=g, device="cuda")
            w["b2"] = 0.05 * torch.randn(spec.f, generator=g, device="cuda")
        layers.append(sffn.Layer.from_weights(w, spec.group_size, spec.act))
        weights.append(w)
    return layers, weights


def _stack_run(sffn, stack, x0, thres, ws=None, masks=None):
    nL, d = stack.n_layers, stack.d
    xs = torch.full((nL, d), float("nan"), device="cuda")
    ys = torch.full((nL, d), float("nan"), device="cuda")
    masks = masks or stack.masks()
    ws = ws if ws is not None else stack.workspace()
    sffn.sffn_stack_decode(stack.handle, x0, xs, ys, thres, masks, ws)
    torch.cuda.synchronize()
    return xs, ys, masks


def _chain_run(sffn, layers, x0, thres):
    """The per-layer calls, x_out chaining the layers."""
    ws = layers[0].workspace()
    out = []
    x = x0.view(1, -1)
    for L in layers:
        m = L.masks()
        y = torch.empty(1, L.d, device="cuda")
        xo = torch.empty(1, L.d, device="cuda")
        sffn.sffn_decode_step(L.handle, x, 1, thres, m, y, xo, ws)
        out.append((m, y, xo))
        x = xo
    torch.cuda.synchronize()
    return out


def _compare(spec, hosts, x0, thres, xs, ys, masks, chain):
    """Oracle per layer (teacher-forced) and the chain where the masks agree.
    Returns the number of layers whose masks equal the chain's."""
    nL, f, G = len(hosts), spec.f, spec.group_size
    same = 0
    x_in = x0.reshape(-1)
    for l in range(nL):
        xs_in = x_in.double().cpu().numpy()
        s = hosts[l].scores(xs_in)
        check_masks(s, thres, G, masks.nmask[l].cpu().numpy(), masks.gmask[l].cpu().numpy(),
                    masks.idx[l].cpu().numpy(), masks.count[l].item())
        gb = words_bits(masks.nmask[l].cpu().numpy(), f)
        check_y(ys[l].cpu().numpy(), hosts[l].ffn(xs_in, gb, spec.act), spec.wdtype, f"y[l={l}]")
        assert torch.equal(xs[l], x_in + ys[l]), l
        if chain is not None:
            m, y, xo = chain[l]
            if torch.equal(m.nmask[0], masks.nmask[l]):
                same += 1
                c = masks.count[l].item()
                assert m.count[0].item() == c
                assert torch.equal(m.gmask[0], masks.gmask[l])
                assert torch.equal(m.idx[0, :c], masks.idx[l, :c])
                if l == 0 or torch.equal(chain[l - 1][2][0], xs[l - 1]):
                    assert torch.equal(y[0], ys[l]), l
                    assert torch.equal(xo[0], xs[l]), l
        x_in = xs[l]
    return same


SHAPES = [
    # d, f, h, G, act, dtype, layers, biases
    (8192, 8192, 1024, 64, "reglu", "bf16", 3, False),      # 70B rows, fewer neurons
    (4096, 11008, 512, 32, "swiglu", "bf16", 4, False),     # 7B SwiGLU shape
    (4096, 16384, 1024, 32, "relu", "f16", 2, True),        # OPT shape, with biases
    (1032, 1088, 72, 64, "reglu", "bf16", 3, True),         # ragged: d / 8 and f / 32 not multiples of the grid
    (1536, 2048, 96, 32, "relu2", "bf16", 2, False),
    (16384, 2048, 64, 32, "relu", "bf16", 2, False),        # 32 KB rows, one per stage
    (64, 64, 8, 32, "swiglu", "f16", 5, True),              # fewer rows and words than blocks
]


@pytest.mark.parametrize("d,f,h,G,act,dt,nL,biases", SHAPES)
def test_stack_against_oracle_and_chain(sffn, d, f, h, G, act, dt, nL, biases):
    spec = W.LayerSpec(name="t", d=d, f=f, h=h, group_size=G, act=act, wdtype=dt, p_mean=0.15, zipf_alpha=1.0)
    layers, weights = _layers(sffn, spec, nL, seed=3, biases=biases)
    hosts = [HostLayer(w, dt) for w in weights]
    stack = sffn.Stack(layers)
    X = W.make_tokens(d, 3, seed=4, kind="ar1", device="cuda")
    same = total = 0
    for t in range(X.shape[0]):
        for thres in (0.0, -0.05):
            x0 = X[t, 0].contiguous()
            xs, ys, masks = _stack_run(sffn, stack, x0, thres)
            chain = _chain_run(sffn, layers, x0, thres)
            same += _compare(spec, hosts, x0, thres, xs, ys, masks, chain)
            total += nL
    assert same >= total - 1, (same, total)
    stack.check_error()


def test_stack_70b_eight_layers(sffn):
    """The full 8-layer 70B-shaped stack, two tokens, the second fed the
    first's output in place (x0 = xs[7])."""
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"]
    nL = spec.layers
    layers = []
    for l in range(nL):
        w = W.make_layer(spec, seed=0, layer=l, device="cuda")
        layers.append(sffn.Layer.from_weights(w, spec.group_size, spec.act))
        del w
    stack = sffn.Stack(layers)
    x0 = W.spec_tokens(spec, 1, seed=0, device="cuda")[0, 0].contiguous()
    ws = stack.workspace()
    xs = torch.empty(nL, spec.d, device="cuda")
    ys = torch.empty(nL, spec.d, device="cuda")
    runs = []
    inp = x0.clone()
    for t in range(2):
        masks = stack.masks()
        src = x0 if t == 0 else xs[nL - 1]       # in place: the previous token's output row
        inp = src.clone()
        sffn.sffn_stack_decode(stack.handle, src, xs, ys, spec.thres, masks, ws)
        torch.cuda.synchronize()
        runs.append((inp, xs.clone(), ys.clone(), masks))
    chain = _chain_run(sffn, layers, runs[1][0], spec.thres)
    for l in range(nL):
        w = W.make_layer(spec, seed=0, layer=l, device="cuda")
        host = HostLayer(w, spec.wdtype)
        del w
        for t, (inp, xs_t, ys_t, masks) in enumerate(runs):
            x_in = inp if l == 0 else xs_t[l - 1]
            xs_in = x_in.double().cpu().numpy()
            s = host.scores(xs_in)
            m = check_masks(s, spec.thres, spec.group_size, masks.nmask[l].cpu().numpy(),
                            masks.gmask[l].cpu().numpy(), masks.idx[l].cpu().numpy(), masks.count[l].item())
            assert abs(m["active"] / spec.f - spec.p_mean) < 0.5 * spec.p_mean
            gb = words_bits(masks.nmask[l].cpu().numpy(), spec.f)
            check_y(ys_t[l].cpu().numpy(), host.ffn(xs_in, gb, spec.act), spec.wdtype, f"y[t={t}, l={l}]")
        del host
    # the second token against the per-layer chain
    inp, xs_t, ys_t, masks = runs[1]
    agree = sum(torch.equal(chain[l][0].nmask[0], masks.nmask[l]) for l in range(nL))
    assert agree >= nL - 1
    if agree == nL:
        assert torch.equal(chain[-1][2][0], xs_t[nL - 1])
    stack.check_error()


@pytest.mark.parametrize("act,dt", [("reglu", "bf16"), ("relu", "f16"), ("swiglu", "bf16")])
def test_stack_all_and_none_active(sffn, act, dt):
    spec = W.LayerSpec(name="t", d=2048, f=4096, h=256, group_size=64, act=act, wdtype=dt, p_mean=0.1,
                       zipf_alpha=1.0)
    layers, weights = _layers(sffn, spec, 2, seed=5)
    stack = sffn.Stack(layers)
    x0 = W.make_tokens(spec.d, 1, seed=6, device="cuda")[0, 0].contiguous()
    xs, ys, masks = _stack_run(sffn, stack, x0, float("-inf"))
    assert (masks.count == spec.f).all() and (masks.nmask == -1).all()
    x_in = x0
    for l in range(2):
        h = HostLayer(weights[l], dt)
        xv = x_in.double().cpu().numpy()
        U, Dn = O.widen(h.up, dt), O.widen(h.down, dt)
        Gt = O.widen(h.gate, dt) if h.gate is not None else None
        check_y(ys[l].cpu().numpy(), O.ffn_dense(xv, U, Gt, Dn, act), dt, f"dense y[{l}]")
        x_in = xs[l]
    xs, ys, masks = _stack_run(sffn, stack, x0, float("inf"))
    assert (masks.count == 0).all() and (masks.nmask == 0).all() and (masks.gmask == 0).all()
    assert (ys == 0).all() and torch.equal(xs[0], x0) and torch.equal(xs[1], x0)
    stack.check_error()


def test_stack_deterministic_and_graph_replay(sffn):
    spec = W.LayerSpec(name="t", d=4096, f=8192, h=512, group_size=32, act="swiglu", wdtype="bf16", p_mean=0.3,
                       zipf_alpha=1.0)
    layers, _ = _layers(sffn, spec, 3, seed=7)
    stack = sffn.Stack(layers)
    x0 = W.make_tokens(spec.d, 1, seed=8, device="cuda")[0, 0].contiguous()
    xs1, ys1, m1 = _stack_run(sffn, stack, x0, 0.0)
    xs2, ys2, m2 = _stack_run(sffn, stack, x0, 0.0)
    assert torch.equal(xs1, xs2) and torch.equal(ys1, ys2) and torch.equal(m1.nmask, m2.nmask)
    # captured in a CUDA graph and replayed: the same results
    ws = stack.workspace()
    xs = torch.empty(3, spec.d, device="cuda")
    ys = torch.empty(3, spec.d, device="cuda")
    masks = stack.masks()
    xin = x0.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sffn.sffn_stack_decode(stack.handle, xin, xs, ys, 0.0, masks, ws, s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sffn.sffn_stack_decode(stack.handle, xin, xs, ys, 0.0, masks, ws)
    xs.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(xs, xs1) and torch.equal(ys, ys1) and torch.equal(masks.nmask, m1.nmask)
    stack.check_error()


def test_stack_argument_checks(sffn):
    spec = W.LayerSpec(name="t", d=256, f=512, h=64, group_size=32, act="relu", wdtype="f16", p_mean=0.2,
                       zipf_alpha=1.0)
    layers, _ = _layers(sffn, spec, 2, seed=9)
    other = sffn.Layer(512, 512, 64, 32, "relu", "f16")
    with pytest.raises(sffn.SffnError) as e:
        sffn.Stack([layers[0], other])
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    f32 = sffn.Layer(256, 512, 64, 32, "relu", "f32")
    with pytest.raises(sffn.SffnError) as e:
        sffn.Stack([f32])
    assert e.value.status == sffn.SFFN_ERR_UNSUPPORTED
    q8 = sffn.Layer(256, 512, 64, 32, "relu", "bf16", ffn_format="q8")
    with pytest.raises(sffn.SffnError) as e:
        sffn.Stack([q8])
    assert e.value.status == sffn.SFFN_ERR_UNSUPPORTED
    stack = sffn.Stack(layers)
    x0 = torch.zeros(spec.d, device="cuda")
    xs = torch.empty(2, spec.d, device="cuda")
    ws = stack.workspace()
    masks = stack.masks()
    with pytest.raises(sffn.SffnError) as e:        # workspace too small
        sffn.sffn_stack_decode(stack.handle, x0, xs, None, 0.0, masks, ws[:-256])
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    with pytest.raises(sffn.SffnError) as e:        # ys overlapping xs
        sffn.sffn_stack_decode(stack.handle, x0, xs, xs, 0.0, masks, ws)
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    with pytest.raises(sffn.SffnError) as e:        # x0 inside xs but not at a row start
        sffn.sffn_stack_decode(stack.handle, xs.view(-1)[4:], xs, None, 0.0, masks, ws)
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    sffn.sffn_stack_decode(stack.handle, x0, xs, None, 0.0, masks, ws)
    stack.check_error()
