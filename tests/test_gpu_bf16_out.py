"""GPU parity of the bf16-output entry point (based_fwd_bf16_out) against the fp64 CPU oracle.

The output contract allows a bf16 output (the kernel-task spec's contract_md: "bf16 or fp32").
Each element must be the fp32 result of the default path rounded to nearest even, so besides the
oracle bar (max|d| <= 2e-2, mean|d| <= 2e-3, relative Frobenius <= 2e-2 against the exact fp64
result) the bf16 output is compared bit for bit with the fp32 output of based_fwd rounded by
torch (round to nearest even) on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_gb300.based import BasedError, based_fwd, based_fwd_bf16_out, workspace_size
from parity_check import assert_all_heads_close
from linear_attention_gb300.inputs import GRADER_WORKLOADS, make_inputs, make_workload

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, REL_FRO = 2e-2, 2e-3, 2e-2

SHAPES = [
    # B, T, H, K, V, seed, scale
    (1, 1, 1, 16, 64, 40, None),
    (2, 63, 2, 8, 128, 41, None),
    (1, 129, 3, 16, 128, 42, 0.2),
    (2, 700, 3, 8, 64, 43, 0.3),
    (1, 1100, 64, 16, 64, 44, None),   # prefixes summed in the forward kernel
    (2, 4096, 8, 16, 128, 45, None),   # prefixes from the scan kernel
    (3, 1000, 5, 8, 128, 46, None),
]


def _check(o_bf16: torch.Tensor, o_f32: torch.Tensor, ref: np.ndarray, what):
    assert o_bf16.dtype == torch.bfloat16
    # the bf16 output is the fp32 output rounded to nearest even, bit for bit
    assert torch.equal(o_bf16.view(torch.int16), o_f32.to(torch.bfloat16).view(torch.int16)), what
    got = o_bf16.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    d = np.abs(got - ref)
    mx, mn, rf = float(d.max()), float(d.mean()), float(np.linalg.norm(d) / np.linalg.norm(ref))
    assert mx <= MAX_ABS and mn <= MEAN_ABS and rf <= REL_FRO, (what, mx, mn, rf)


@pytest.mark.parametrize("B,T,H,K,V,seed,scale", SHAPES,
                         ids=[f"B{c[0]}T{c[1]}H{c[2]}K{c[3]}V{c[4]}" for c in SHAPES])
def test_bf16_output_matches_oracle(B, T, H, K, V, seed, scale, cuda_device):
    q, k, v = make_inputs(B, T, H, K, V, seed)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    o16 = based_fwd_bf16_out(qd, kd, vd, scale=scale)
    o32 = based_fwd(qd, kd, vd, scale=scale)
    torch.cuda.synchronize()
    sc = oracle.default_scale(K) if scale is None else float(np.float32(scale))
    ref, _ = oracle.chunked(q, k, v, sc, chunk=64)
    _check(o16, o32, ref, (B, T, H, K, V))


def test_bf16_output_caller_workspace_and_events(cuda_device):
    B, T, H, K, V = 2, 3000, 3, 16, 128
    q, k, v = [t.to(cuda_device) for t in make_inputs(B, T, H, K, V, 47)]
    ws = torch.empty(max(workspace_size(B, T, H, K, V), 16), dtype=torch.uint8, device=cuda_device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e1.record()
    o1 = based_fwd_bf16_out(q, k, v)
    o2 = based_fwd_bf16_out(q, k, v, workspace=ws, events=(e0, e1))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert e0.elapsed_time(e1) > 0
    with pytest.raises(BasedError):
        based_fwd_bf16_out(q, k, v, workspace=ws[:1])


def test_bf16_output_not_written_past_end(cuda_device):
    B, T, H, K, V = 1, 200, 3, 16, 64
    q, k, v = [t.to(cuda_device) for t in make_inputs(B, T, H, K, V, 48)]
    n = B * T * H * V
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device=cuda_device)
    based_fwd_bf16_out(q, k, v, out=buf[:n].view(B, T, H, V))
    torch.cuda.synchronize()
    assert torch.all(buf[n:] == 7.0)


@pytest.mark.parametrize("name", ["grader2", "grader5"])
def test_bf16_output_grader_shape(name, cuda_device):
    """A full grading shape (B=8, H=32, T up to 16384): the bf16 output is the fp32 output rounded
    to nearest even, bit for bit, and every element is within the bar of the oracle."""
    w = GRADER_WORKLOADS[name]
    q, k, v = make_workload(w)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    o16 = based_fwd_bf16_out(qd, kd, vd, scale=w.scale)
    o32 = based_fwd(qd, kd, vd, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    del o32
    sc = oracle.default_scale(w.K) if w.scale is None else float(np.float32(w.scale))
    assert_all_heads_close(o16.float().cpu().numpy(), q, k, v, sc, f"{name} bf16 output")
