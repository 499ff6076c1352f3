"""GB300-native Based (2nd-order Taylor linear attention) causal forward pass.

The compute runs in hand-written sm_103a CUDA kernels behind a C-ABI shared library
(``include/based.h``); ``linear_attention_gb300.based`` is a thin ctypes binding to it.
"""
import importlib

__all__ = ["based_fwd", "based_fwd_host"]


def __getattr__(name):
    # The binding is imported lazily so that the input generators can be used without the
    # CUDA library being built.
    if name in ("based_fwd", "based_fwd_host"):
        return getattr(importlib.import_module(".based", __name__), name)
    raise AttributeError(name)
