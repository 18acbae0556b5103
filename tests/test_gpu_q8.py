"""8-bit and 4-bit quantized FFN rows (SFFN_FFN_Q8, SFFN_FFN_Q4) through the
C ABI: each weight is a code times one float32 scale per neuron (up and gate
rows, down columns), the predictor stays 16-bit. Masks bit-exact outside the
score band, y against the oracle's quantized sparse FFN on the GPU's own mask;
the packed 4-bit rows equal the oracle's encoding of the codes.
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


def _check_tokens(sffn, spec, L, host, X):
    masks, ws = L.masks(), L.workspace()
    y = torch.empty(1, spec.d, device="cuda")
    for t in range(X.shape[0]):
        sffn.sffn_decode_step(L.handle, X[t], 1, spec.thres, masks, y, None, ws)
        xs = X[t][0].double().cpu().numpy()
        check_masks(host.scores(xs), spec.thres, spec.group_size, masks.nmask[0].cpu().numpy(),
                    masks.gmask[0].cpu().numpy(), masks.idx[0].cpu().numpy(), masks.count[0].item())
        gb = words_bits(masks.nmask[0].cpu().numpy(), spec.f)
        check_y(y[0].cpu().numpy(), host.ffn(xs, gb, spec.act), spec.wdtype, f"y[{t}]")
    L.check_error()


SHAPES = [
    # d, f, h, G, act, predictor dtype (d a multiple of 16)
    (1024, 2048, 128, 32, "relu", "bf16"),
    (2048, 1024, 64, 64, "reglu", "f16"),
    (528, 960, 96, 32, "swiglu", "bf16"),
    (4096, 2048, 256, 32, "relu2", "bf16"),
]


@pytest.mark.parametrize("d,f,h,G,act,dt", SHAPES)
def test_q8_small_shapes(sffn, d, f, h, G, act, dt):
    spec = W.LayerSpec(name="q8", d=d, f=f, h=h, group_size=G, act=act, wdtype=dt, p_mean=0.12, zipf_alpha=1.0,
                       ffn_q8=True)
    L, w, host = make_layer(spec, seed=1)
    assert host.q8
    _check_tokens(sffn, spec, L, host, W.make_tokens(d, 2, seed=2, device="cuda"))


def test_q8_full_size_70b_layer(sffn):
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_q8_8l"]
    L, w, host = make_layer(spec, seed=0)
    _check_tokens(sffn, spec, L, host, W.make_tokens(spec.d, 2, seed=0, kind=spec.seq, device="cuda"))


def test_q8_rules(sffn):
    spec = W.LayerSpec(name="q8", d=512, f=1024, h=64, group_size=32, act="reglu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0, ffn_q8=True)
    w = W.make_layer(spec, seed=0, device="cuda")
    L = sffn.Layer.from_weights(w, 32, "reglu", max_batch=4)
    wf = W.make_layer(W.spec_replace(spec, ffn_q8=False), seed=0, device="cuda")
    with pytest.raises(sffn.SffnError) as e:        # the plain pack refuses 8-bit layers
        sffn.sffn_layer_pack(L.handle, wf["W1"], None, wf["W2"], None, wf["up"], wf["gate"], wf["down"], None)
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    L16 = sffn.Layer.from_weights(wf, 32, "reglu")
    with pytest.raises(sffn.SffnError) as e:        # and the 8-bit pack refuses 16-bit layers
        L16.pack(w)
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    x = torch.zeros(4, spec.d, device="cuda")
    y = torch.empty(4, spec.d, device="cuda")
    with pytest.raises(sffn.SffnError) as e:        # batched calls need 16-bit rows
        sffn.sffn_decode_step(L.handle, x, 4, 0.0, L.masks(4), y, None, L.workspace(4))
    assert e.value.status == sffn.SFFN_ERR_UNSUPPORTED
    pv = L.packed()
    assert pv.up_scale and pv.gate_scale and pv.down_scale
    assert not L16.packed().up_scale


SHAPES_Q4 = [
    # d a multiple of 32
    (1024, 2048, 128, 32, "relu", "bf16"),
    (2048, 1024, 64, 64, "reglu", "f16"),
    (544, 960, 96, 32, "swiglu", "bf16"),
    (4096, 2048, 256, 32, "relu2", "bf16"),
]


@pytest.mark.parametrize("d,f,h,G,act,dt", SHAPES_Q4)
def test_q4_small_shapes(sffn, d, f, h, G, act, dt):
    spec = W.LayerSpec(name="q4", d=d, f=f, h=h, group_size=G, act=act, wdtype=dt, p_mean=0.12, zipf_alpha=1.0,
                       ffn_q4=True)
    L, w, host = make_layer(spec, seed=1)
    assert host.q8 and host.qbits == 4 and L.ffn_format == "q4"
    _check_tokens(sffn, spec, L, host, W.make_tokens(d, 2, seed=2, device="cuda"))


def test_q4_full_size_70b_layer(sffn):
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_q4_8l"]
    L, w, host = make_layer(spec, seed=0)
    _check_tokens(sffn, spec, L, host, W.make_tokens(spec.d, 2, seed=0, kind=spec.seq, device="cuda"))


def test_q4_packed_rows_match_the_oracle_encoding(sffn):
    spec = W.LayerSpec(name="q4", d=256, f=512, h=64, group_size=32, act="reglu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0, ffn_q4=True)
    L, w, host = make_layer(spec, seed=3)
    pv = L.packed()
    perm = w["perm"].cpu().numpy()
    for ptr, codes in ((pv.up, w["up_q"].cpu().numpy()), (pv.gate, w["gate_q"].cpu().numpy()),
                       (pv.downT, w["down_q"].cpu().numpy().T)):
        got = sffn.view_device(ptr, (spec.f, spec.d // 2), torch.uint8).cpu().numpy()
        assert (got == O.pack_q4(codes[perm])).all()
    ups = sffn.view_device(pv.up_scale, (spec.f,), torch.float32).cpu().numpy()
    assert (ups == w["up_s"].cpu().numpy()[perm]).all()


def test_q4_rules(sffn):
    spec = W.LayerSpec(name="q4", d=512, f=1024, h=64, group_size=32, act="reglu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0, ffn_q4=True)
    w = W.make_layer(spec, seed=0, device="cuda")
    L = sffn.Layer.from_weights(w, 32, "reglu")
    with pytest.raises(sffn.SffnError) as e:        # the 8-bit pack refuses 4-bit layers
        sffn.sffn_layer_pack_q8(L.handle, w["W1"], None, w["W2"], None, w["up_q"], w["up_s"], w["gate_q"],
                                w["gate_s"], w["down_q"], w["down_s"], None)
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
    bad = w["up_q"].clone()
    bad[3, 5] = 9                                   # outside [-8, 7]
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_layer_pack_q4(L.handle, w["W1"], None, w["W2"], None, bad, w["up_s"], w["gate_q"], w["gate_s"],
                                w["down_q"], w["down_s"], None)
    assert e.value.status == sffn.SFFN_ERR_DEVICE
    L.check_error()                                 # reported by the pack call, so cleared
    with pytest.raises(sffn.SffnError) as e:        # d must be a multiple of 32
        sffn.Layer(528, 1024, 64, 32, "reglu", "bf16", 1, "q4")
    assert e.value.status == sffn.SFFN_ERR_INVALID_ARG
