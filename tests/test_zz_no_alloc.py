"""The allocation-free entry point (based_fwd_noalloc, scratch in a fixed device array) against
the regular entry point (based_fwd, library-owned workspace), both called through the C ABI.

Calls in a row with different shapes and inputs: a later one must not see anything an earlier one
left in the shared scratch array. Every shape splits heads across CTAs, so the aggregate kernel
(and the scan, where the plan needs it) runs and the scratch is used. Tolerance: the parity bar of
the GPU tests (max |diff| <= 2e-2, mean |diff| <= 2e-3); where both entry points use the same
plan they agree exactly, and the last shape checks the smaller plan the scratch forces.
"""
import ctypes

import pytest
import torch

from linear_attention_gb300.based import device_status, kernel_count, library, workspace_size
from linear_attention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
SHAPES = [  # B, T, H, K, V, seed
    (2, 2048, 8, 16, 64, 41),
    (1, 3000, 6, 8, 128, 42),
    # based_fwd cuts this shape's aggregate pass into 288 pieces (one slot each), which would not
    # fit the 16 MiB scratch at 82,560 bytes per slot: the no-allocation call keeps one slot per
    # range and sums in another order
    (2, 16384, 32, 16, 128, 43),
]


def _call(fn, q, k, v, o):
    B, T, H, K = q.shape
    V = v.shape[-1]
    rc = fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), B, T, H, K, V, ctypes.c_float(-1.0),
            ctypes.c_void_p(o.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, library().based_strerror(rc).decode()


def test_noalloc_matches_based_fwd_twice(cuda_device):
    L = library()
    device_status(0, clear=True)
    for B, T, H, K, V, seed in SHAPES:
        assert workspace_size(B, T, H, K, V) > 0 and kernel_count(B, T, H, K, V) >= 2
        q, k, v = (x.to(cuda_device) for x in make_inputs(B, T, H, K, V, seed))
        o_ref = torch.empty(B, T, H, V, dtype=torch.float32, device=cuda_device)
        o_na = torch.full_like(o_ref, float("nan"))
        _call(L.based_fwd, q, k, v, o_ref)
        _call(L.based_fwd_noalloc, q, k, v, o_na)
        torch.cuda.synchronize()
        assert torch.isfinite(o_na).all()
        d = (o_na - o_ref).abs()
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, (B, T, H, K, V)
    assert device_status(0, clear=True) == 0
