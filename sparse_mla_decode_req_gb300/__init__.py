"""GB300-native sparse MLA decode over an fp8_ds_mla paged latent cache.

The compute lives in ``libsmd.so`` (hand-written CUDA for sm_103a, C ABI declared in
``include/smd.h``).  ``sparse_mla_decode_req_gb300.api`` is a thin ctypes binding with
the same names; importing this package does not load the library, so the synthetic
input module (``synth``) can be used on machines without a GPU.
"""
import importlib

__all__ = ["api", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
