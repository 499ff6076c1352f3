"""Seeded synthetic inputs for the Based causal forward pass.

This module holds no arithmetic of the method: it only names the workloads and draws q, k, v.
Both the CUDA path's tests and the CPU oracle consume what it returns.

Recipe (mirrors the ``_mk`` input generator of the "based_forward.py" kernel-task spec): q, k of
shape (B,T,H,K) and v of shape (B,T,H,V), each i.i.d. standard normal drawn in that order from one
generator seeded with ``seed``, stored as bfloat16. The spec draws on a CUDA generator; here a
CPU ``torch.Generator`` is used so that every run, with or without a GPU, sees the same values.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    seed: int
    scale: Optional[float]  # None means the default K ** -0.5

    @property
    def shape(self):
        return (self.B, self.T, self.H, self.K, self.V)


# The five Based forward workloads: (B, T, H, K, V), seed, scale.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 512, 2, 8, 64, 0, None),
    "mid": Workload("mid", 2, 2048, 16, 16, 64, 1, 0.25),
    "headline": Workload("headline", 4, 4096, 16, 16, 64, 2, None),
    "long": Workload("long", 1, 16384, 16, 16, 128, 3, None),
    "ragged": Workload("ragged", 8, 3000, 12, 8, 128, 4, 0.3),
}

# The shape regime the "based_forward.py" spec grades in (its grader_shapes list; regime_md:
# B 4-8, T 8192-16384, H 16-32, K in {8, 16}, V in {64, 128}), with the same input recipe.
GRADER_WORKLOADS = {
    "grader1": Workload("grader1", 4, 16384, 32, 16, 128, 101, None),
    "grader2": Workload("grader2", 8, 8192, 32, 16, 128, 102, None),
    "grader3": Workload("grader3", 8, 16384, 16, 16, 128, 103, None),
    "grader4": Workload("grader4", 8, 16384, 32, 16, 64, 104, None),
    "grader5": Workload("grader5", 8, 16384, 32, 8, 128, 105, None),
}


def make_inputs(B: int, T: int, H: int, K: int, V: int, seed: int, device="cpu"):
    """q, k, v ~ N(0,1) in bfloat16, drawn in the order q, k, v from one seeded CPU generator."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn(B, T, H, K, dtype=torch.bfloat16, generator=gen)
    k = torch.randn(B, T, H, K, dtype=torch.bfloat16, generator=gen)
    v = torch.randn(B, T, H, V, dtype=torch.bfloat16, generator=gen)
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def make_workload(w: Workload, device="cpu"):
    return make_inputs(w.B, w.T, w.H, w.K, w.V, w.seed, device=device)
