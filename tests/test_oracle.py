"""Pins for the CPU oracle (no GPU).

Each pin checks the oracle against something other than itself: hand-worked values derived from
the spec's definition, closed forms of special cases, exact identities and invariants that the
"based_forward.py" kernel-task spec states, brute force on tiny inputs, and a textbook routine
(causal softmax attention) in the limit where the Taylor polynomial approaches exp. The last test
plants plausible mistakes in the oracle's C source and requires every one to fail some pin.
"""
import json
import math
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from linear_attention_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "based_handworked.json")
ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "based_oracle.c")


def _rand(B, T, H, K, V, seed):
    q, k, v = make_inputs(B, T, H, K, V, seed)
    return q.double().numpy(), k.double().numpy(), v.double().numpy()


def _relfro(a, b):
    return float(np.linalg.norm((a - b).ravel()) / np.linalg.norm(b.ravel()))


# ------------------------------------------------------------------------------------------------
# Pins, written as functions of an oracle library handle so that the mutation test can run them
# against a deliberately broken build.
# ------------------------------------------------------------------------------------------------

def pin_golden(L):
    """Hand-worked cases (tests/golden/based_handworked.json), both evaluation forms."""
    d = json.load(open(GOLDEN))
    for c in d["cases"]:
        B, T, H, K, V = c["B"], c["T"], c["H"], c["K"], c["V"]
        q = np.array(c["q"], dtype=np.float64).reshape(B, T, H, K)
        k = np.array(c["k"], dtype=np.float64).reshape(B, T, H, K)
        v = np.array(c["v"], dtype=np.float64).reshape(B, T, H, V)
        num = np.array(c["num"], dtype=np.float64)
        den = np.array(c["den"], dtype=np.float64)
        want = num / (den[:, None] + 1e-6)
        for form in ("direct", "chunked1", "chunked2", "chunked256"):
            if form == "direct":
                o, dn = oracle.direct(q, k, v, c["scale"], L=L)
            else:
                o, dn = oracle.chunked(q, k, v, c["scale"], chunk=int(form[7:]), L=L)
            np.testing.assert_allclose(o.reshape(T, V), want, rtol=1e-13, atol=1e-13,
                                       err_msg=f"{c['name']} {form}")
            np.testing.assert_allclose(dn.reshape(T), den, rtol=1e-13, atol=1e-13,
                                       err_msg=f"{c['name']} {form} den")


def pin_phi_identity(L):
    """phi(q).phi(k) = 1 + q.k + (q.k)^2/2 (spec_md, 'Why this is not an O(T^2) op')."""
    rng = np.random.default_rng(11)
    for K in (1, 3, 8, 16):
        assert oracle.feature_len(K, L) == 1 + K + K * K
        for _ in range(20):
            x, y = rng.standard_normal(K), rng.standard_normal(K)
            d = float(x @ y)
            got = float(oracle.phi(x, L) @ oracle.phi(y, L))
            assert abs(got - (1 + d + d * d / 2)) <= 1e-12 * max(1.0, abs(got)), (K, got)


def pin_phi_basis(L):
    """phi(e_a) = 1 at slot 0, 1 at slot 1+a, 1/sqrt(2) at slot 1+K+a*K+a, zero elsewhere."""
    for K in (8, 16):
        for a in range(K):
            e = np.zeros(K)
            e[a] = 1.0
            want = np.zeros(1 + K + K * K)
            want[0] = 1.0
            want[1 + a] = 1.0
            want[1 + K + a * K + a] = 2.0 ** -0.5
            np.testing.assert_allclose(oracle.phi(e, L), want, rtol=0, atol=1e-15)


def pin_chunked_equals_direct(L):
    """Brute force: the chunked feature-map form equals the O(T^2) double sum."""
    for (B, T, H, K, V, C, seed) in [(2, 37, 3, 8, 5, 8, 1), (1, 130, 2, 16, 64, 64, 2),
                                     (2, 64, 1, 16, 3, 16, 3), (1, 5, 2, 8, 4, 2, 4)]:
        q, k, v = _rand(B, T, H, K, V, seed)
        sc = K ** -0.5
        od, dd = oracle.direct(q, k, v, sc, L=L)
        oc, dc = oracle.chunked(q, k, v, sc, chunk=C, L=L)
        assert np.abs(od - oc).max() <= 1e-12 * max(1.0, np.abs(od).max())
        assert np.abs(dd - dc).max() <= 1e-12 * dd.max()


def pin_chunk_invariance(L):
    """The answer does not depend on the chunk length (spec_md, last paragraph)."""
    B, T, H, K, V = 1, 300, 2, 16, 8
    q, k, v = _rand(B, T, H, K, V, 5)
    ref, _ = oracle.chunked(q, k, v, 0.25, chunk=T, L=L)
    for C in (1, 7, 64, 128, 256):
        o, _ = oracle.chunked(q, k, v, 0.25, chunk=C, L=L)
        assert np.abs(o - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max()), C


def pin_denominator_positive(L):
    """1 + s + s^2/2 = ((1+s)^2 + 1)/2 >= 1/2, so den_i >= (i+1)/2 (precision_md)."""
    q, k, v = _rand(2, 200, 2, 8, 4, 6)
    q *= 3.0  # wide spread of scores, many negative
    for form in ("direct", "chunked"):
        if form == "direct":
            _, den = oracle.direct(q, k, v, 1.0, L=L)
        else:
            _, den = oracle.chunked(q, k, v, 1.0, chunk=64, L=L)
        lower = (np.arange(200) + 1) / 2.0
        assert np.all(den >= lower[None, :, None] - 1e-12)


def pin_zero_query_prefix_mean(L):
    """q = 0 (or k = 0) gives s = 0, A = 1: o_i is the prefix sum of v over (i+1) + 1e-6."""
    B, T, H, K, V = 1, 150, 2, 16, 6
    _, k, v = _rand(B, T, H, K, V, 7)
    zeros = np.zeros((B, T, H, K))
    want = np.cumsum(v, axis=1) / (np.arange(1, T + 1)[None, :, None, None] + 1e-6)
    for qq, kk in ((zeros, k), (k, zeros)):
        for form in ("direct", "chunked"):
            if form == "direct":
                o, _ = oracle.direct(qq, kk, v, 0.7, L=L)
            else:
                o, _ = oracle.chunked(qq, kk, v, 0.7, chunk=32, L=L)
            np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)


def pin_softmax_limit(L):
    """As the scores shrink, 1 + s + s^2/2 = exp(s) - s^3/6 + O(s^4), so the output approaches
    causal softmax attention within a bound set by max|s|^3 (a weighted-average perturbation)."""
    B, T, H, K, V = 1, 96, 2, 16, 8
    q, k, v = _rand(B, T, H, K, V, 8)
    scale = 0.004
    s = scale * np.einsum("bihd,bjhd->bhij", q, k)
    smax = float(np.abs(s).max())
    assert smax < 0.2
    mask = np.tril(np.ones((T, T), dtype=bool))
    w = np.where(mask, np.exp(s), 0.0)
    soft = np.einsum("bhij,bjhd->bihd", w / w.sum(-1, keepdims=True), v)
    delta = smax ** 3 / 6 * math.exp(2 * smax)  # bound on |A/exp(s) - 1|
    bound = 2 * delta / (1 - delta) * np.abs(v).max() + 4e-6 * np.abs(v).max()
    for form in ("direct", "chunked"):
        if form == "direct":
            o, _ = oracle.direct(q, k, v, scale, L=L)
        else:
            o, _ = oracle.chunked(q, k, v, scale, chunk=32, L=L)
        assert np.abs(o - soft).max() <= bound, (np.abs(o - soft).max(), bound)


def pin_head_layout(L):
    """Each (b, h) head is an independent problem: the batched result equals the result of the
    head sliced out on its own (catches mixed-up B/H/T strides)."""
    B, T, H, K, V = 2, 40, 3, 8, 4
    q, k, v = _rand(B, T, H, K, V, 9)
    for form in ("direct", "chunked"):
        if form == "direct":
            o, _ = oracle.direct(q, k, v, 0.35, L=L)
        else:
            o, _ = oracle.chunked(q, k, v, 0.35, chunk=16, L=L)
        for b in range(B):
            for h in range(H):
                sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
                if form == "direct":
                    oh, _ = oracle.direct(q[sl], k[sl], v[sl], 0.35, L=L)
                else:
                    oh, _ = oracle.chunked(q[sl], k[sl], v[sl], 0.35, chunk=16, L=L)
                np.testing.assert_allclose(o[sl], oh, rtol=1e-14, atol=1e-14)


def pin_linear_in_v(L):
    """Numerator is linear in v and the denominator does not involve v."""
    B, T, H, K, V = 1, 70, 2, 8, 5
    q, k, v1 = _rand(B, T, H, K, V, 10)
    _, _, v2 = _rand(B, T, H, K, V, 11)
    o1, _ = oracle.chunked(q, k, v1, 0.3, chunk=16, L=L)
    o2, _ = oracle.chunked(q, k, v2, 0.3, chunk=16, L=L)
    o3, _ = oracle.chunked(q, k, 2.0 * v1 - 3.0 * v2, 0.3, chunk=16, L=L)
    np.testing.assert_allclose(o3, 2.0 * o1 - 3.0 * o2, rtol=1e-11, atol=1e-12)


def pin_feature_permutation(L):
    """Permuting the K features of q and k together leaves every score, hence o, unchanged."""
    B, T, H, K, V = 1, 90, 2, 16, 4
    q, k, v = _rand(B, T, H, K, V, 12)
    perm = np.random.default_rng(3).permutation(K)
    o, _ = oracle.chunked(q, k, v, 0.25, chunk=32, L=L)
    op, _ = oracle.chunked(q[..., perm], k[..., perm], v, 0.25, chunk=32, L=L)
    np.testing.assert_allclose(op, o, rtol=1e-12, atol=1e-13)


PINS = [pin_golden, pin_phi_identity, pin_phi_basis, pin_chunked_equals_direct,
        pin_chunk_invariance, pin_denominator_positive, pin_zero_query_prefix_mean,
        pin_softmax_limit, pin_head_layout, pin_linear_in_v, pin_feature_permutation]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.lib())


# ------------------------------------------------------------------------------------------------
# The correctness gate must reject the two mistakes the spec names (spec_md, precision_md).
# ------------------------------------------------------------------------------------------------

def _direct_variant(q, k, v, scale, order=2, normalise=True):
    s = scale * np.einsum("bihd,bjhd->bhij", q, k)
    A = 1.0 + s + (0.5 * s * s if order == 2 else 0.0)
    T = q.shape[1]
    A = A * np.tril(np.ones((T, T)))
    num = np.einsum("bhij,bjhd->bihd", A, v)
    if not normalise:
        return num
    return num / (A.sum(-1).transpose(0, 2, 1)[..., None] + 1e-6)


def test_gate_rejects_first_order_and_missing_normaliser():
    B, T, H, K, V = 1, 512, 2, 16, 64
    q, k, v = _rand(B, T, H, K, V, 13)
    sc = oracle.default_scale(K)
    ref, _ = oracle.chunked(q, k, v, sc, chunk=256)
    np.testing.assert_allclose(_direct_variant(q, k, v, sc), ref, rtol=1e-10, atol=1e-12)
    assert _relfro(_direct_variant(q, k, v, sc, order=1), ref) > 2e-2
    assert _relfro(_direct_variant(q, k, v, sc, normalise=False), ref) > 10.0


# ------------------------------------------------------------------------------------------------
# Planted mistakes: each source mutation of the oracle must fail at least one pin.
# ------------------------------------------------------------------------------------------------

MUTANTS = {
    "direct_first_order": ("const double A = 1.0 + s + s * s / 2.0;", "const double A = 1.0 + s;"),
    "chunked_full_square": ("const double A = 1.0 + s + 0.5 * s * s;",
                            "const double A = 1.0 + s + s * s;"),
    "phi_no_sqrt2": ("out[1 + K + a * K + b] = x[a] * x[b] * inv_sqrt2;",
                     "out[1 + K + a * K + b] = x[a] * x[b];"),
    "direct_strict_causal": ("for (int j = 0; j <= i; ++j) {", "for (int j = 0; j < i; ++j) {"),
    "chunked_strict_causal": ("for (int j = 0; j <= r; ++j) {", "for (int j = 0; j < r; ++j) {"),
    "direct_no_normaliser": ("for (int e = 0; e < c->V; ++e) num[e] = num[e] / (den + 1e-6);",
                             "for (int e = 0; e < c->V; ++e) num[e] = num[e];"),
    "direct_scale_on_k_too": ("dot += (c->scale * qi[a]) * kj[a];",
                              "dot += (c->scale * qi[a]) * (c->scale * kj[a]);"),
    "chunked_state_transposed": ("num[e] += pq[p] * S[(int64_t)p * V + e];",
                                 "num[e] += pq[p] * S[(int64_t)e * P + p];"),
    "chunked_z_squared": ("z[p] += pk[p];", "z[p] += pk[p] * pk[p];"),
    "head_index_swapped": ("int b = bh / H, h = bh % H;", "int h = bh / H, b = bh % H;"),
    "chunked_guard_inside": ("orow[e] = num[e] / (den + 1e-6);", "orow[e] = num[e] / den + 1e-6;"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="based_oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = os.path.join(mutant_dir, f"{name}.c")
    open(path, "w").write(src.replace(old, new))
    so = oracle.compile_oracle(path, os.path.join(mutant_dir, f"lib{name}.so"))
    L = oracle.load_library(so)
    caught = []
    for pin in PINS:
        try:
            pin(L)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
