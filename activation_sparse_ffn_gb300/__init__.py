"""Activation-sparse FFN decode on one GB300 (sm_103a CUDA behind a C ABI).

``activation_sparse_ffn_gb300.sffn`` is the binding of the C library
``libsffn.so``; importing it raises if the library has not been built.
``activation_sparse_ffn_gb300.workload`` draws seeded synthetic inputs.
"""

__all__ = ["sffn", "workload"]


def __getattr__(name):
    if name in ("sffn", "workload"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
