"""One-layer-ahead prediction and the B = 1 grid settings, through the C ABI.

KAIROX (问题与动机, observation on adjacent layers) notes that consecutive layers
see near-identical inputs, so the active set of layer l + 1 can be predicted
from layer l's input while layer l's FFN runs. The library computes both
with its existing calls: sffn_predict(layer l + 1, x_l) on a second stream,
overlapping sffn_forward(layer l, x_l) on the first, each on its own share of
the SMs (sffn_layer_set_grid). Parity: layer l + 1's masks equal the oracle
predictor of layer l + 1 applied to the GPU's layer-l input (bit-exact
outside the score band), and each y equals the oracle FFN on the GPU's own
mask (teacher forcing). Recall against the exact masks is reported.
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


def _num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def test_layers_of_different_shapes_interleave(sffn):
    """Creating a smaller layer must not break a larger one created earlier
    (the kernels' shared-memory limits are process-wide)."""
    big = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"], f=4096, tam_capacity=None)
    small = W.WORKLOADS["relu_d512_f2048_fp32"]
    A, _, hostA = make_layer(big, seed=0)
    xA = W.make_tokens(big.d, 1, seed=1, kind="ar1", device="cuda")[0]
    B_, _, hostB = make_layer(small, seed=0)
    xB = W.make_tokens(small.d, 1, seed=1, device="cuda")[0]
    for L, host, spec, x in ((A, hostA, big, xA), (B_, hostB, small, xB), (A, hostA, big, xA)):
        m, ws = L.masks(), L.workspace()
        y = torch.empty(1, spec.d, device="cuda")
        sffn.sffn_decode_step(L.handle, x, 1, spec.thres, m, y, None, ws)
        xs = x[0].double().cpu().numpy()
        gb = words_bits(m.nmask[0].cpu().numpy(), spec.f)
        check_y(y[0].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype)
        L.check_error()


def test_grid_settings(sffn):
    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"], f=8192, tam_capacity=None)
    L, w, host = make_layer(spec, seed=0)
    x = W.make_tokens(spec.d, 1, seed=3, kind="ar1", device="cuda")[0]
    ref_m, ws = L.masks(), L.workspace()
    ref_y = torch.empty(1, spec.d, device="cuda")
    sffn.sffn_decode_step(L.handle, x, 1, spec.thres, ref_m, ref_y, None, ws)
    n = _num_sms()
    xs = x[0].double().cpu().numpy()
    for fb, sb in ((n - 48, 48), (n // 2, 7), (n, 1), (0, 0)):
        L.set_grid(fb, sb)
        m = L.masks()
        y = torch.empty(1, spec.d, device="cuda")
        sffn.sffn_decode_step(L.handle, x, 1, spec.thres, m, y, None, L.workspace())
        for k in ("nmask", "gmask", "idx", "count"):
            assert torch.equal(getattr(m, k), getattr(ref_m, k)), (fb, sb, k)
        gb = words_bits(m.nmask[0].cpu().numpy(), spec.f)
        check_y(y[0].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype, f"grid {fb}/{sb}")
    for bad in ((-1, 0), (n + 1, 0), (0, n + 1)):
        with pytest.raises(sffn.SffnError) as e:
            L.set_grid(*bad)
        assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    L.check_error()


def lookahead_step(sffn, layers, x0, masks, y_out, xbufs, ws_main, ws_side, side, thres, saved=None):
    """One token through the stack with one-layer-ahead prediction: layer 0 is
    predicted from its own input; layer l + 1 from x_l on `side` while layer l's
    FFN runs on the current stream. Returns the last layer's x_out. `saved`
    (optional list) receives (x_l, y_l) copies per layer."""
    main = torch.cuda.current_stream()
    nL = len(layers)
    sffn.sffn_predict(layers[0].handle, x0, 1, thres, masks[0], ws_side, main)
    x = x0
    for l in range(nL):
        ev_p = None
        if l + 1 < nL:
            ev_x = torch.cuda.Event()
            ev_x.record(main)
            side.wait_event(ev_x)
            sffn.sffn_predict(layers[l + 1].handle, x, 1, thres, masks[l + 1], ws_side, side)
            ev_p = torch.cuda.Event()
            ev_p.record(side)
        xo = xbufs[l % 2]
        sffn.sffn_forward(layers[l].handle, x, 1, masks[l], y_out, xo, ws_main, main)
        if saved is not None:
            saved.append((x.clone(), y_out.clone()))
        if ev_p is not None:
            main.wait_event(ev_p)
        x = xo
    return x


def test_lookahead_stack_matches_oracle(sffn):
    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"], f=8192, tam_capacity=None)
    nL, T = 3, 3
    made = [make_layer(spec, seed=0, layer=l) for l in range(nL)]
    layers = [m[0] for m in made]
    hosts = [m[2] for m in made]
    n = _num_sms()
    for L in layers:
        L.set_grid(n - 48, 48)
    masks = [L.masks() for L in layers]
    ws_main, ws_side = layers[0].workspace(), layers[0].workspace()
    side = torch.cuda.Stream()
    y = torch.empty(1, spec.d, device="cuda")
    xbufs = (torch.empty(1, spec.d, device="cuda"), torch.empty(1, spec.d, device="cuda"))
    X = W.make_tokens(spec.d, T, seed=5, kind="ar1", device="cuda")
    recall = []
    for t in range(T):
        saved = []
        snap = []
        # masks are overwritten by later tokens: keep this token's views per layer
        lookahead_step(sffn, layers, X[t], masks, y, xbufs, ws_main, ws_side, side, spec.thres, saved)
        torch.cuda.synchronize()
        for l in range(nL):
            snap.append({k: getattr(masks[l], k).clone() for k in ("nmask", "gmask", "idx", "count")})
        for l in range(nL):
            x_l, y_l = (a[0].double().cpu().numpy() for a in saved[l])
            src = x_l if l == 0 else saved[l - 1][0][0].double().cpu().numpy()   # predictor input
            s = hosts[l].scores(src)
            v = snap[l]
            check_masks(s, spec.thres, spec.group_size, v["nmask"][0].cpu().numpy(), v["gmask"][0].cpu().numpy(),
                        v["idx"][0].cpu().numpy(), v["count"][0].item())
            gb = words_bits(v["nmask"][0].cpu().numpy(), spec.f)
            check_y(y_l, hosts[l].ffn(x_l, gb, spec.act), spec.wdtype, f"y[t={t}, l={l}]")
            if l > 0:
                exact = O.active_from_scores(hosts[l].scores(x_l), spec.thres)
                recall.append((gb & exact).sum() / max(1, exact.sum()))
    print(f"look-ahead recall of the exact active set: mean {np.mean(recall):.3f}, min {np.min(recall):.3f}")
    assert np.mean(recall) > 0.5
    for L in layers:
        L.check_error()
