"""The allocation-free entry point (based_fwd_noalloc, scratch in a fixed device array) against
the regular entry point (based_fwd, library-owned workspace), both called through the C ABI.

Some callers cannot allocate device memory while they run: a serving loop whose memory is planned
up front by its own allocator, or code that must not take the device-wide synchronisation that
cudaMalloc / cudaFree can cause. based_fwd_noalloc is for them. This file checks that it gives
based_fwd's result and that it allocates nothing:
  - calls in a row with different shapes and inputs: a later call must not see anything an
    earlier one left in the shared scratch array. Every shape but the last splits heads across
    CTAs with the aggregate pass, so the scratch is used; the last one's ranges run lead-ins
    instead (one kernel, no scratch);
  - the last shape's regular plan needs more than the fixed scratch, so the no-allocation call
    takes the smaller plan (one slot per range) and sums in another order;
  - the free device memory is the same before and after the calls (after one small warm-up call
    per kernel variant, which loads the kernels' code).
Tolerance: the parity bar of the GPU tests (max |diff| <= 2e-2, mean |diff| <= 2e-3); where both
entry points use the same plan they agree exactly.
"""
import ctypes

import pytest
import torch

from linear_attention_gb300.based import device_status, kernel_count, library, workspace_size
from linear_attention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024  # BASED_NOALLOC_SCRATCH_BYTES in include/based.h
SHAPES = [  # B, T, H, K, V, seed
    (1, 8192, 8, 16, 64, 41),
    (1, 3000, 6, 8, 128, 42),
    # based_fwd cuts this shape's aggregate pass into 66 pieces per head lane, 4 lanes, one
    # 82,560-byte slot each (21.8 MB), which do not fit the fixed scratch
    (8, 8192, 32, 16, 128, 43),
]
LEAD_IN = (2, 2048, 8, 16, 64, 48)
WARMUP = [(1, 1024, 2, 16, 64, 44), (1, 1024, 2, 8, 128, 45), (1, 1024, 2, 16, 128, 46),
          (1, 2048, 4, 16, 128, 47)]


def _call(fn, q, k, v, o):
    B, T, H, K = q.shape
    V = v.shape[-1]
    rc = fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), B, T, H, K, V, ctypes.c_float(-1.0),
            ctypes.c_void_p(o.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, library().based_fwd_strerror(rc).decode()


def test_noalloc_matches_based_fwd_in_a_row(cuda_device):
    L = library()
    device_status(0, clear=True)
    assert workspace_size(*SHAPES[-1][:5]) > NOALLOC_SCRATCH_BYTES
    cases = []
    for B, T, H, K, V, seed in SHAPES + [LEAD_IN]:
        if (B, T, H, K, V, seed) == LEAD_IN:
            assert workspace_size(B, T, H, K, V) == 0 and kernel_count(B, T, H, K, V) == 1
        else:
            assert workspace_size(B, T, H, K, V) > 0 and kernel_count(B, T, H, K, V) >= 2
        q, k, v = (x.to(cuda_device) for x in make_inputs(B, T, H, K, V, seed))
        o_ref = torch.empty(B, T, H, V, dtype=torch.float32, device=cuda_device)
        _call(L.based_fwd, q, k, v, o_ref)
        cases.append((q, k, v, o_ref, torch.full_like(o_ref, float("nan"))))
    for B, T, H, K, V, seed in WARMUP:  # loads the code of every kernel variant the calls use
        q, k, v = (x.to(cuda_device) for x in make_inputs(B, T, H, K, V, seed))
        _call(L.based_fwd_noalloc, q, k, v, torch.empty(B, T, H, V, device=cuda_device))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(cuda_device)[0]
    for q, k, v, _, o_na in cases:
        _call(L.based_fwd_noalloc, q, k, v, o_na)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(cuda_device)[0] == free_before, "based_fwd_noalloc allocated"
    for (q, k, v, o_ref, o_na), shape in zip(cases, SHAPES + [LEAD_IN]):
        assert torch.isfinite(o_na).all(), shape
        d = (o_na - o_ref).abs()
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, shape
    assert device_status(0, clear=True) == 0
