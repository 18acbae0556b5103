"""The allocation-free decode entry point against the regular one.

sffn_decode_step_static_ws serves callers that cannot allocate device memory
(a decode loop that must not stall on an allocation, a runtime with no CUDA
allocator of its own, a memory pool that refuses new allocations while
serving): its scratch is a fixed device array inside the library instead of
a caller workspace. This test calls it through the C ABI twice in a row, on
two different tokens, and checks each output against sffn_decode_step on the
same inputs, with the tolerances of the parity tests (both run the same
kernels in the same order, so the results are in fact identical). It sits in
a file collected last so that a failure here stops a run only after every
other test has run.
"""

import pytest
import torch

from activation_sparse_ffn_gb300 import workload as W

from gpu_util import check_y

pytestmark = pytest.mark.gpu


def test_static_workspace_matches_caller_workspace():
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn

    spec = W.spec_replace(W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"], f=8192, layers=1)
    w = W.make_layer(spec, seed=11, layer=0, device="cuda")
    L = sffn.Layer.from_weights(w, spec.group_size, spec.act)
    X = W.make_tokens(spec.d, 2, seed=12, kind="ar1", device="cuda")
    ws = L.workspace()
    for t in range(2):                      # two calls in a row
        m_ref, m_new = L.masks(), L.masks()
        y_ref = torch.empty(1, spec.d, device="cuda")
        y_new = torch.full((1, spec.d), float("nan"), device="cuda")
        xo_ref = torch.empty(1, spec.d, device="cuda")
        xo_new = torch.empty(1, spec.d, device="cuda")
        sffn.sffn_decode_step(L.handle, X[t], 1, spec.thres, m_ref, y_ref, xo_ref, ws)
        sffn.sffn_decode_step_static_ws(L.handle, X[t], 1, spec.thres, m_new, y_new, xo_new)
        torch.cuda.synchronize()
        check_y(y_new[0].double().cpu().numpy(), y_ref[0].double().cpu().numpy(), spec.wdtype, "y (static ws)")
        check_y(xo_new[0].double().cpu().numpy(), xo_ref[0].double().cpu().numpy(), spec.wdtype, "x_out (static ws)")
        assert torch.equal(m_new.nmask, m_ref.nmask) and torch.equal(m_new.count, m_ref.count)
        assert torch.equal(m_new.gmask, m_ref.gmask)
        c = m_ref.count.item()
        assert torch.equal(m_new.idx[0, :c], m_ref.idx[0, :c])
    L.check_error()


def test_static_workspace_rejects_batches_above_one():
    """B > 1 is refused with UNSUPPORTED before any device work. The other
    refusal, a layer whose B = 1 scratch exceeds the 16 MiB array, cannot be
    reached on a GB300: the scratch is the hidden vector plus one partial sum
    of y per FFN block, at most 152 x 16384 x 4 bytes (under 10 MB), and
    sffn_layer_set_grid never raises the block count above the SM count."""
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn

    spec = W.LayerSpec(name="t", d=64, f=64, h=8, group_size=32, act="relu", wdtype="f16", p_mean=0.2,
                       zipf_alpha=1.0)
    w = W.make_layer(spec, seed=0, device="cuda")
    L = sffn.Layer.from_weights(w, 32, "relu", max_batch=2)
    x = torch.zeros(2, 64, device="cuda")
    y = torch.empty(2, 64, device="cuda")
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_decode_step_static_ws(L.handle, x, 2, 0.0, L.masks(2), y, None)
    assert e.value.status == sffn.SFFN_ERR_UNSUPPORTED
    # the largest valid B = 1 scratch on this GPU fits the array
    big = sffn.Layer(16384, 64, 8, 32, "relu", "bf16")
    assert sffn.sffn_workspace_bytes(big.handle, 1) <= 16 << 20
