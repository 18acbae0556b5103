"""The C ABI without a GPU: the library builds and loads, exports every
function include/sffn.h declares, and its host-side argument checks return
the documented status codes before any device work."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sffn.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from activation_sparse_ffn_gb300 import sffn
    return sffn


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?[\s\*]+([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("typedef")))


def test_header_declares_the_calls():
    names = declared_functions()
    for must in ("sffn_predict", "sffn_forward", "sffn_decode_step", "tam_update", "tam_adapt",
                 "sffn_layer_create", "sffn_layer_pack", "sffn_workspace_bytes"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing
    assert sorted(lib.EXPORTS) == declared_functions()


def test_status_strings(lib):
    assert lib.status_string(0) == "SFFN_OK"
    assert lib.status_string(4) == "SFFN_ERR_TIMEOUT"
    assert lib.status_string(99) == "SFFN_ERR_UNKNOWN"
    assert lib.version().startswith("sffn")


@pytest.mark.parametrize("kw,ok", [
    (dict(d=8192, f=28672, h=1024, group_size=64, act="reglu", wdtype="bf16"), True),
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype="f32"), True),
    (dict(d=4096, f=11008, h=512, group_size=32, act="swiglu", wdtype="bf16", max_batch=32), True),
    (dict(d=8192, f=32768, h=1024, group_size=32, act="relu", wdtype="f16"), True),
    (dict(d=8, f=32, h=8, group_size=32, act="relu", wdtype="bf16"), True),
    (dict(d=100, f=2048, h=64, group_size=32, act="relu", wdtype="f32"), False),     # d % 8
    (dict(d=16384, f=2048, h=64, group_size=32, act="relu", wdtype="f32"), False),   # row > 32 KB
    (dict(d=512, f=2000, h=64, group_size=32, act="relu", wdtype="f32"), False),     # f % G
    (dict(d=512, f=2048, h=64, group_size=48, act="relu", wdtype="f32"), False),     # G
    (dict(d=512, f=65600, h=64, group_size=32, act="relu", wdtype="f16"), False),    # > 1024 groups
    (dict(d=512, f=2048, h=12, group_size=32, act="relu", wdtype="f32"), False),     # h % 8
    (dict(d=512, f=2048, h=1024, group_size=32, act="relu", wdtype="f32"), False),   # predictor row > 2 KB
    (dict(d=512, f=2048, h=1024, group_size=32, act="relu", wdtype="bf16"), True),
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype="f32", max_batch=33), False),
    (dict(d=512, f=2048, h=64, group_size=32, act=7, wdtype="f32"), False),
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype=9), False),
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype="bf16", ffn_format="q8"), True),
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype="f32", ffn_format="q8"), False),   # fp32 predictor
    (dict(d=520, f=2048, h=64, group_size=32, act="relu", wdtype="bf16", ffn_format="q8"), False),  # d % 16
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype="bf16", ffn_format=5), False),
    (dict(d=512, f=2048, h=64, group_size=32, act="relu2", wdtype="bf16"), True),
    (dict(d=512, f=2048, h=64, group_size=32, act=4, wdtype="bf16"), False),
    (dict(d=512, f=2048, h=64, group_size=32, act="reglu", wdtype="f16", ffn_format="q4"), True),
    (dict(d=528, f=2048, h=64, group_size=32, act="relu", wdtype="bf16", ffn_format="q4"), False),  # d % 32
    (dict(d=528, f=2048, h=64, group_size=32, act="relu", wdtype="bf16", ffn_format="q8"), True),   # d % 16 is enough
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype="f32", ffn_format="q4"), False),   # fp32 predictor
    (dict(d=16384, f=2048, h=64, group_size=32, act="relu", wdtype="bf16"), True),    # 32 KB rows
    (dict(d=16392, f=2048, h=64, group_size=32, act="relu", wdtype="f16"), False),    # d > 16384
    (dict(d=512, f=32, h=64, group_size=64, act="relu", wdtype="f32"), False),        # f < G
    (dict(d=512, f=65536, h=64, group_size=64, act="relu", wdtype="f16"), True),      # exactly 1024 groups
    (dict(d=512, f=2048, h=64, group_size=32, act="relu", wdtype="f32", max_batch=0), False),
    (dict(d=512, f=2048, h=512, group_size=32, act="relu", wdtype="f32"), True),      # 2 KB predictor rows
])
def test_validate(lib, kw, ok):
    desc = lib.make_desc(**kw)
    rc = lib.sffn_layer_validate(desc)
    assert rc == (lib.SFFN_OK if ok else lib.SFFN_ERR_INVALID_ARG), lib.last_error()


def test_null_handles_are_rejected_on_the_host(lib):
    L = lib._lib
    m = lib.MasksC()
    assert L.sffn_predict(None, None, 1, 0.0, ctypes.byref(m), None, 0, None) == lib.SFFN_ERR_INVALID_ARG
    assert "NULL" in lib.last_error()
    assert L.sffn_forward(None, None, 1, ctypes.byref(m), None, None, None, 0, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_decode_step(None, None, 1, 0.0, ctypes.byref(m), None, None, None, 0, None) == lib.SFFN_ERR_INVALID_ARG
    o = lib.TamOutputsC()
    assert L.sffn_decode_step_tam(None, None, 0, None, 1, 0.0, ctypes.byref(m), None, None, None, 0, 0.9, 0.01, 1,
                                  ctypes.byref(o), None) == lib.SFFN_ERR_INVALID_ARG
    assert L.tam_update(None, 0, 1, None, 1, 0.9, 0.01, 1, ctypes.byref(o), None) == lib.SFFN_ERR_INVALID_ARG
    assert L.tam_adapt(None, 0, 1, None, 0.01, 0.8, 0.99, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_layer_pack(None, None, None, None, None, None, None, None, None, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_workspace_bytes(None, 1) == 0
    assert L.sffn_layer_check_error(None, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_selftest_wait_timeout(None, 10, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_layer_set_next(None, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_layer_set_grid(None, 0, 0) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_layer_set_l2_resident(None, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_layer_set_zero_skip(None, 1, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_layer_set_batch_path(None, 0) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_layer_batch_arm(None, 2) == -1
    assert L.sffn_stack_create(None, 1, ctypes.byref(ctypes.c_void_p())) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_stack_workspace_bytes(None) == 0
    assert L.sffn_stack_check_error(None, None) == lib.SFFN_ERR_INVALID_ARG
    assert L.sffn_stack_decode(None, None, None, None, 0.0, ctypes.byref(m), None, 0, None) == lib.SFFN_ERR_INVALID_ARG
    L.sffn_stack_destroy(None)
    out = ctypes.c_void_p()
    assert L.sffn_layer_create(None, ctypes.byref(out)) == lib.SFFN_ERR_INVALID_ARG
    bad = lib.make_desc(100, 2048, 64, 32, "relu", "f32")
    assert L.sffn_layer_create(ctypes.byref(bad), ctypes.byref(out)) == lib.SFFN_ERR_INVALID_ARG
    assert out.value is None
    for args in [(0, 10, 0.9), (1, 0, 0.9), (1, 2000, 0.9), (1, 10, 1.0), (1, 10, 0.0)]:
        assert L.tam_create(*args, ctypes.byref(out)) == lib.SFFN_ERR_INVALID_ARG
    L.sffn_layer_destroy(None)
    L.tam_destroy(None)
