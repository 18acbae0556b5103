"""The 32-layer SwiGLU decode loop of the 7B-shaped workload, through the C ABI:
every layer's mask views against the oracle (teacher-forced on the GPU's own
layer input), per-layer momentum with the adaptive lambda step (KAIROX 核心方法
items 4 and 5) bit-exact every token, and a topic shift half way that re-draws
every layer's group ranks (new W2, re-packed).

The residual stream is x_{l+1} = x_l + y_l. A gated FFN grows roughly with the
square of its input, so without the normalisation a transformer block applies
before its FFN the stream overflows within a few of the 32 layers; the
harness therefore feeds each layer x_l / rms(x_l) (no learned scale), a
stand-in for the rest of the block, not a step of the FFN path.
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


def test_swiglu_32_layer_loop_with_adaptive_lambda_and_topic_shift(sffn):
    spec = W.WORKLOADS["swiglu7b_d4096_f11008_bf16_32l"]
    nL, G, f, ng = spec.layers, spec.group_size, spec.f, spec.n_groups
    T, shift = 8, 4
    K = spec.capacity
    eps = np.float32(spec.tam_eps)
    y_checks = {(0, shift - 1), (nL - 1, shift - 1), (0, shift), (nL - 1, shift)}

    layers, weights, W1h, W2h = [], [], [], []
    for l in range(nL):
        w = W.make_layer(spec, seed=0, layer=l, device="cuda")
        layers.append(sffn.Layer.from_weights(w, G, spec.act))
        weights.append(w)
        W1h.append(O.widen(W.stored_numpy(w["W1"]), spec.wdtype))
        W2h.append(O.widen(W.stored_numpy(w["W2"]), spec.wdtype))
    perms = [w["perm"].cpu().numpy().astype(np.int64) for w in weights]
    ffn_host = {l: HostLayer(weights[l], spec.wdtype) for l in (0, nL - 1)}

    tam = sffn.Tam(nL, ng, spec.tam_lambda)
    outs = sffn.TamOutputs(nL, ng, K)
    gw = (ng + 31) // 32
    gm_all = torch.zeros(nL, gw, dtype=torch.int32, device="cuda")
    stalls = W.make_stall_bits(T, nL, seed=0)
    s_ref = np.zeros((nL, ng), dtype=np.float32)
    prev = np.zeros((nL, ng), dtype=bool)
    lam = np.full(nL, spec.tam_lambda, dtype=np.float32)

    X = W.make_tokens(spec.d, T, seed=0, kind=spec.seq, device="cuda")
    masks = [L.masks() for L in layers]
    ws = layers[0].workspace()
    y = torch.empty(1, spec.d, device="cuda")
    xa, xb = torch.empty(1, spec.d, device="cuda"), torch.empty(1, spec.d, device="cuda")
    sc = torch.empty(nL, ng, device="cuda")
    la = torch.empty(nL, device="cuda")
    active = np.zeros((T, nL, f), dtype=bool)
    band_total = 0

    for t in range(T):
        if t == shift:
            # topic shift: each layer's group ranks are redrawn (new W2 offsets), the layer re-packed
            for l in range(nL):
                w = dict(weights[l])
                w["W2"] = W.make_w2_topic(spec, 0, l, 1, w["W1"], w["perm"])
                layers[l].pack(w)
                weights[l] = w
                W2h[l] = O.widen(W.stored_numpy(w["W2"]), spec.wdtype)
            torch.cuda.synchronize()
        resid = X[t].clone()
        for l in range(nL):
            x = resid / torch.sqrt((resid * resid).mean())
            xo = (xa, xb)[l % 2]
            sffn.sffn_decode_step(layers[l].handle, x, 1, spec.thres, masks[l], y, xo, ws)
            xs = x[0].double().cpu().numpy()
            s = O.predictor_scores(W2h[l], O.predictor_hidden(W1h[l], xs))[perms[l]]
            m = check_masks(s, spec.thres, G, masks[l].nmask[0].cpu().numpy(), masks[l].gmask[0].cpu().numpy(),
                            masks[l].idx[0].cpu().numpy(), masks[l].count[0].item())
            band_total += m["band"]
            active[t, l] = words_bits(masks[l].nmask[0].cpu().numpy(), f)
            assert abs(active[t, l].mean() - spec.p_mean) < 0.1, (t, l)
            if (l, t) in y_checks:
                check_y(y[0].cpu().numpy(), ffn_host[l].ffn(xs, active[t, l], spec.act), spec.wdtype,
                        f"y[t={t}, l={l}]")
            assert torch.equal(xo, x + y)
            gm_all[l].copy_(masks[l].gmask[0])
            resid = resid + y
        # momentum of every layer from this token's group masks, then the lambda step
        sffn.tam_update(tam.handle, 0, nL, gm_all, gw, -1.0, spec.tam_eps, K, outs)
        sffn.tam_adapt(tam.handle, 0, nL, torch.from_numpy(stalls[t]).cuda(), spec.anb_alpha, spec.anb_lo,
                       spec.anb_hi)
        sffn.tam_get_state(tam.handle, sc, la, None)
        scores_gpu, lam_gpu = sc.cpu().numpy(), la.cpu().numpy()
        for l in range(nL):
            ga = words_bits(gm_all[l].cpu().numpy(), ng)
            r = O.tam_update(s_ref[l], prev[l], ga, lam[l], eps, K)
            s_ref[l], prev[l] = r["scores"], r["resident"]
            k = r["topk"].shape[0]
            assert np.array_equal(outs.topk[l, :k].cpu().numpy(), r["topk"]), (t, l)
            assert np.array_equal(words_bits(outs.resident[l].cpu().numpy(), ng), r["resident"]), (t, l)
            assert np.array_equal(words_bits(outs.changed[l].cpu().numpy(), ng), r["changed"]), (t, l)
            lam[l] = O.anb_step(lam[l], bool(stalls[t, l]), spec.anb_alpha, spec.anb_lo, spec.anb_hi)
        assert np.array_equal(scores_gpu, s_ref), t
        assert np.array_equal(lam_gpu, lam), t

    # the shift re-draws which neurons fire: consecutive tokens agree less across it than within a topic
    def jac(a, b):
        return (a & b).sum() / max(1, (a | b).sum())
    j = np.array([[jac(active[t, l], active[t + 1, l]) for l in range(nL)] for t in range(T - 1)]).mean(axis=1)
    within = np.delete(j, shift - 1)
    assert j[shift - 1] < 0.9 * within.min(), j
    # about 10 of 11008 scores per layer-token fall in the excluded band; bound it at 0.2%
    assert band_total < 0.002 * f * nL * T
    for L in layers:
        L.check_error()
    sffn.tam_check_error(tam.handle)
