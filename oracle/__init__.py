"""CPU oracle for the Based causal forward pass (fp64).

TEST INFRASTRUCTURE ONLY: this package may be imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``, and by nothing else.
The product path (``linear_attention_gb300``) never imports, links or runs it, and it shares no
code with the CUDA library.

The arithmetic lives in ``based_oracle.c`` (plain C, fp64, loops), which restates the
"based_forward.py" kernel-task spec (spec_md and reference_src); this module only builds it with
gcc and marshals numpy arrays through ctypes.

Parity status: every function here is pinned by ``tests/test_oracle.py`` (brute force on tiny
inputs, the feature-map identity, chunk-size invariance, closed-form special cases, the
softmax limit, hand-worked golden cases and source mutations that the pins must catch).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "based_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libbased_oracle.so")
_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc (portable flags only)."""
    cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared", src,
           "-o", out, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library next to its source if it is missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            compile_oracle()
    return _LIB_PATH


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    lib.based_oracle_feature_len.argtypes = [ctypes.c_int]
    lib.based_oracle_feature_len.restype = ctypes.c_int
    lib.based_oracle_phi.argtypes = [dp, ctypes.c_int, dp]
    lib.based_oracle_phi.restype = None
    lib.based_oracle_direct_rows.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [
        ctypes.c_double, ip, ctypes.c_int64, dp, dp, ctypes.c_int]
    lib.based_oracle_direct_rows.restype = ctypes.c_int
    lib.based_oracle_chunked.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_int, ip, ctypes.c_int64, dp, dp, ctypes.c_int]
    lib.based_oracle_chunked.restype = ctypes.c_int
    lib.based_oracle_default_threads.argtypes = []
    lib.based_oracle_default_threads.restype = ctypes.c_int
    return lib


def load_library(path: str):
    """Load an oracle shared library from ``path`` (tests use this for source mutants)."""
    return _bind(ctypes.CDLL(path))


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load_library(_LIB_PATH)
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: bf16 -> fp64 is exact
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def default_threads(L=None) -> int:
    return int((L or lib()).based_oracle_default_threads())


def feature_len(K: int, L=None) -> int:
    return int((L or lib()).based_oracle_feature_len(K))


def phi(x, L=None) -> np.ndarray:
    """phi(x) = [1, x, vec(x (x) x)/sqrt(2)] for a 1-D x."""
    L = L or lib()
    x = _f64(x).reshape(-1)
    out = np.empty(feature_len(x.size, L), dtype=np.float64)
    L.based_oracle_phi(_dptr(x), x.size, _dptr(out))
    return out


def direct_rows(q, k, v, scale: float, pairs, nthreads: int = 0, L=None):
    """Direct O(T^2) definition at chosen (bh, i) pairs; returns (o_rows (n,V), den_rows (n,))."""
    L = L or lib()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, H, K = q.shape
    V = v.shape[-1]
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    n = pairs.shape[0]
    o = np.empty((n, V), dtype=np.float64)
    den = np.empty((n,), dtype=np.float64)
    rc = L.based_oracle_direct_rows(_dptr(q), _dptr(k), _dptr(v), B, T, H, K, V, float(scale),
                                    _iptr(pairs), n, _dptr(o), _dptr(den), nthreads)
    if rc != 0:
        raise ValueError("based_oracle_direct_rows rejected its arguments")
    return o, den


def direct(q, k, v, scale: float, nthreads: int = 0, L=None):
    """Direct definition over every (head, row): returns (o (B,T,H,V), den (B,T,H))."""
    q = _f64(q)
    B, T, H, _ = q.shape
    V = _f64(v).shape[-1]
    bh, t = np.meshgrid(np.arange(B * H), np.arange(T), indexing="ij")
    pairs = np.stack([bh.reshape(-1), t.reshape(-1)], axis=1)
    o, den = direct_rows(q, k, v, scale, pairs, nthreads, L)
    o = o.reshape(B, H, T, V).transpose(0, 2, 1, 3)
    den = den.reshape(B, H, T).transpose(0, 2, 1)
    return np.ascontiguousarray(o), np.ascontiguousarray(den)


def chunked(q, k, v, scale: float, chunk: int = 256, heads=None, nthreads: int = 0, L=None):
    """Chunked feature-map form. With heads=None returns (o (B,T,H,V), den (B,T,H)); with a list
    of flattened head indices bh = b*H + h returns (o (n,T,V), den (n,T))."""
    L = L or lib()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if heads is None:
        hs = np.arange(B * H, dtype=np.int64)
    else:
        hs = np.ascontiguousarray(np.asarray(heads, dtype=np.int64).reshape(-1))
    n = hs.size
    o = np.empty((n, T, V), dtype=np.float64)
    den = np.empty((n, T), dtype=np.float64)
    rc = L.based_oracle_chunked(_dptr(q), _dptr(k), _dptr(v), B, T, H, K, V, float(scale),
                                int(chunk), _iptr(hs), n, _dptr(o), _dptr(den), nthreads)
    if rc != 0:
        raise ValueError("based_oracle_chunked rejected its arguments")
    if heads is None:
        o = np.ascontiguousarray(o.reshape(B, H, T, V).transpose(0, 2, 1, 3))
        den = np.ascontiguousarray(den.reshape(B, H, T).transpose(0, 2, 1))
    return o, den


def default_scale(K: int) -> float:
    """scale=None means K ** -0.5 (contract_md); the fp32 value is what a kernel receives."""
    return float(np.float32(K ** -0.5))
