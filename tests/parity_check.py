"""Comparison of a CUDA output with the fp64 chunked oracle over every element (shared by the GPU
parity tests). Bar (the Based forward workload definition): max|o_gpu - o_oracle| <= 2e-2 and
mean|o_gpu - o_oracle| <= 2e-3 in fp32 output units, and the relative Frobenius error against the
spec's correctness gate (2e-2). With BASED_PARITY_LOG set to a file path, each comparison appends
its error figures to that file as a JSON line."""
import json
import os

import numpy as np

import oracle

MAX_ABS, MEAN_ABS, REL_FRO = 2e-2, 2e-3, 2e-2


def _errors(o_gpu: np.ndarray, ref: np.ndarray):
    d = np.abs(o_gpu.astype(np.float64) - ref)
    return float(d.max()), float(d.mean()), float(np.linalg.norm(d) / np.linalg.norm(ref))


def _log(what, mx, mn, rf, n):
    path = os.environ.get("BASED_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": str(what), "max_abs": mx, "mean_abs": mn, "rel_fro": rf,
                                "elements": int(n)}) + "\n")


def _assert_close(o_gpu, ref, what):
    mx, mn, rf = _errors(o_gpu, ref)
    _log(what, mx, mn, rf, o_gpu.size)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    assert mx <= MAX_ABS and mn <= MEAN_ABS and rf <= REL_FRO, (what, mx, mn, rf)
    return mx, mn, rf


def assert_all_heads_close(o_gpu, q, k, v, scale, what, batch=32):
    """Every element of o_gpu (B,T,H,V) against the chunked oracle, computed over all B*H heads in
    batches of `batch` heads (bounded host memory on the largest shapes)."""
    o_gpu = np.asarray(o_gpu)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    B, T, H, V = o_gpu.shape
    qn, kn, vn = (np.ascontiguousarray(t.double().numpy()) for t in (q, k, v))
    mx, s_abs, s_d2, s_r2 = 0.0, 0.0, 0.0, 0.0
    for h0 in range(0, B * H, batch):
        heads = list(range(h0, min(B * H, h0 + batch)))
        ref, _ = oracle.chunked(qn, kn, vn, scale, chunk=256, heads=heads)
        got = np.stack([o_gpu[h // H, :, h % H, :] for h in heads]).astype(np.float64)
        d = np.abs(got - ref)
        mx = max(mx, float(d.max()))
        s_abs += float(d.sum())
        s_d2 += float((d * d).sum())
        s_r2 += float((ref * ref).sum())
    mn, rf = s_abs / o_gpu.size, float(np.sqrt(s_d2 / s_r2))
    _log(what, mx, mn, rf, o_gpu.size)
    assert mx <= MAX_ABS and mn <= MEAN_ABS and rf <= REL_FRO, (what, mx, mn, rf)
    return mx, mn, rf
