"""Actual-activation zero-skip of the B = 1 sparse FFN, through the C ABI.

With zero-skip on, the FFN reads the transposed-down row of a predicted-active
neuron only if its activation h is non-zero. y must equal the oracle FFN on the
GPU's own mask (and, bit for bit up to the sign of zero, the same call without
zero-skip); the number of rows read must equal the oracle's count of non-zero
activations, up to the neurons whose pre-activation is so close to zero that
fp32 and fp64 may disagree on its sign.
"""

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gb300 import workload as W
from oracle import sffn_oracle as O

from gpu_util import check_y, make_layer, words_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn as mod
    return mod


def _decode(sffn, L, x, thres):
    masks = L.masks(1)
    ws = L.workspace(1)
    y = torch.full((L.d,), float("nan"), device="cuda")
    xo = torch.empty(L.d, device="cuda")
    sffn.sffn_decode_step(L.handle, x[None], 1, thres, masks, y[None], xo[None], ws)
    torch.cuda.synchronize()
    return masks, y, xo


def _rows_reference(host, xs, bits, act):
    """Oracle count of down rows read, and how many neurons sit in the sign band."""
    orig = host.perm[np.flatnonzero(bits)] if host.perm is not None else np.flatnonzero(bits)
    U = O.widen(host.up[orig], host.dt)
    G = O.widen(host.gate[orig], host.dt) if host.gate is not None else None
    D = O.widen(host.down[:, orig], host.dt)
    ones = np.ones(orig.shape[0], dtype=bool)
    y, n = O.ffn_sparse_zero_skip(xs, U, G, D, act, ones)
    u = U @ xs
    near = np.abs(u) < 1e-4 * max(np.abs(u).max(initial=0.0), 1e-30)
    if G is not None:
        g = G @ xs
        near |= np.abs(g) < 1e-4 * max(np.abs(g).max(initial=0.0), 1e-30)
    return y, n, int(near.sum())


SHAPES = [
    # d, f, h, G, act, dtype
    (1024, 2048, 128, 32, "relu", "f16"),
    (1024, 4096, 256, 64, "reglu", "bf16"),
    (768, 2048, 192, 64, "relu2", "bf16"),
    (1024, 2048, 128, 32, "swiglu", "bf16"),
    (512, 1024, 64, 32, "reglu", "f32"),
]


@pytest.mark.parametrize("d,f,h,G,act,dt", SHAPES)
def test_zero_skip_matches_oracle_and_counts_rows(sffn, d, f, h, G, act, dt):
    spec = W.LayerSpec(name="t", d=d, f=f, h=h, group_size=G, act=act, wdtype=dt, p_mean=0.15, zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=21)
    rows = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for t in range(3):
        x = W.make_tokens(d, 1, seed=30 + t, device="cuda")[0, 0].contiguous()
        L.set_zero_skip(False)
        m0, y0, _ = _decode(sffn, L, x, 0.0)
        L.set_zero_skip(True, rows)
        m1, y1, xo1 = _decode(sffn, L, x, 0.0)
        assert torch.equal(m0.nmask, m1.nmask) and torch.equal(m0.idx, m1.idx) and torch.equal(m0.count, m1.count)
        # a skipped row would only have added h * w = 0
        assert torch.equal(y1 + 0.0, y0 + 0.0)
        assert torch.equal(xo1, x + y1)
        xs = x.double().cpu().numpy()
        bits = words_bits(m1.nmask[0].cpu().numpy(), f)
        y_ref, n_ref, band = _rows_reference(host, xs, bits, act)
        check_y(y1.cpu().numpy(), y_ref, dt)
        n = int(rows.item())
        assert abs(n - n_ref) <= band, (n, n_ref, band)
        assert 0 <= n <= int(bits.sum())
    L.check_error()


def test_zero_skip_reglu_reads_fewer_rows_and_off_writes_nothing(sffn):
    spec = W.LayerSpec(name="t", d=1024, f=4096, h=128, group_size=64, act="reglu", wdtype="bf16", p_mean=0.2,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=5)
    rows = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    x = W.make_tokens(spec.d, 1, seed=6, device="cuda")[0, 0].contiguous()
    L.set_zero_skip(True, rows)
    m, _, _ = _decode(sffn, L, x, 0.0)
    n, active = int(rows.item()), int(m.count[0].item())
    assert 0 < n < active   # independent gates: some predicted neurons clamp to zero
    L.set_zero_skip(False, rows)   # off: the pointer is dropped
    rows.fill_(-1)
    _decode(sffn, L, x, 0.0)
    assert int(rows.item()) == -1
    L.check_error()


def test_zero_skip_full_size_70b_layer(sffn):
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"]
    L, w, host = make_layer(spec, seed=0, layer=0)
    rows = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    L.set_zero_skip(True, rows)
    x = W.make_tokens(spec.d, 1, seed=1, kind=spec.seq, device="cuda")[0, 0].contiguous()
    m, y, _ = _decode(sffn, L, x, spec.thres)
    xs = x.double().cpu().numpy()
    bits = words_bits(m.nmask[0].cpu().numpy(), spec.f)
    y_ref, n_ref, band = _rows_reference(host, xs, bits, spec.act)
    check_y(y.cpu().numpy(), y_ref, spec.wdtype)
    assert abs(int(rows.item()) - n_ref) <= band
    L.check_error()


def test_zero_skip_ignored_by_batches(sffn):
    spec = W.LayerSpec(name="t", d=1024, f=2048, h=128, group_size=32, act="relu", wdtype="bf16", p_mean=0.1,
                       zipf_alpha=1.0)
    L, w, host = make_layer(spec, seed=9, max_batch=8)
    X = W.make_tokens(spec.d, 1, seed=10, batch=4, device="cuda")[0]
    out = []
    for on in (False, True):
        L.set_zero_skip(on)
        masks = L.masks(4)
        y = torch.empty(4, spec.d, device="cuda")
        sffn.sffn_decode_step(L.handle, X, 4, 0.0, masks, y, None, L.workspace(4))
        torch.cuda.synchronize()
        out.append(y)
    assert torch.equal(out[0], out[1])
    L.check_error()
