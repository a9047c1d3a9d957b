"""Pins for the float64 oracle: closed forms, invariants, special cases.

None of these retypes the oracle's formulas.  Newton-Schulz is checked against
its action on singular values (numpy's SVD, then the scalar quintic), against
exact rational arithmetic in the 1x1 case, against matrices whose singular
values are all equal, and against equivariances.  Momentum is checked on small
integers, the hyperball on its norm invariant and fixed points, bfloat16
rounding against torch's conversion.  The last block plants mistakes in copies
of the oracle and shows that the pins catch each one.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import muonh as om

COEFFS = (3.4445, -4.7750, 2.0315)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _quintic(s, coeffs, steps):
    a, b, c = coeffs
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def _ns_by_svd(m, steps, coeffs, eps):
    """Newton-Schulz through its action on singular values."""
    m = np.asarray(m, np.float64)
    u, sig, vt = np.linalg.svd(m, full_matrices=False)
    x_sig = sig / (np.sqrt(np.sum(m * m)) + eps)
    return (u * _quintic(x_sig, coeffs, steps)) @ vt


def _rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300))


def _ns_svd_error(ns, shapes=((1, 1), (3, 7), (7, 3), (8, 4), (16, 16), (5, 40)), seed=0):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for shape in shapes:
        m = rng.standard_normal(shape)
        for steps in (1, 2, 5):
            worst = max(worst, _rel(ns(m, steps, COEFFS, 1e-7), _ns_by_svd(m, steps, COEFFS, 1e-7)))
    return worst


# --- Newton-Schulz -----------------------------------------------------------

def test_ns_matches_singular_value_polynomial():
    assert _ns_svd_error(om.newton_schulz) < 1e-12


def test_ns_rank_deficient_matches_svd():
    rng = np.random.default_rng(1)
    for shape, rank in (((12, 20), 3), ((20, 12), 2), ((9, 9), 1)):
        m = rng.standard_normal((shape[0], rank)) @ rng.standard_normal((rank, shape[1]))
        got = om.newton_schulz(m, 5, COEFFS, 1e-7)
        assert _rel(got, _ns_by_svd(m, 5, COEFFS, 1e-7)) < 1e-11
        assert np.linalg.matrix_rank(got, tol=1e-8) == rank


def test_ns_scalar_exact_rational():
    # 1x1: x0 = m / (|m| + eps), then x <- a x + b x^3 + c x^5, in exact rationals.
    for m in (0.75, -3.0, 1e-3):
        eps = 1e-7
        x = Fraction(m) / (abs(Fraction(m)) + Fraction(eps))
        a, b, c = (Fraction(v) for v in COEFFS)
        for _ in range(5):
            x = a * x + b * x ** 3 + c * x ** 5
        got = om.newton_schulz(np.array([[m]]), 5, COEFFS, eps)[0, 0]
        assert abs(got - float(x)) <= 4e-16 * abs(float(x))


def test_ns_equal_singular_values_closed_form():
    # M = alpha * Q with orthonormal rows: every singular value of X0 is
    # alpha / (alpha*sqrt(s) + eps), so O = p^k(that) * Q exactly.
    rng = np.random.default_rng(2)
    for s, l in ((4, 4), (6, 10), (10, 6)):
        q, _ = np.linalg.qr(rng.standard_normal((max(s, l), min(s, l))))
        q = q.T if s <= l else q        # orthonormal rows (wide) or columns (tall)
        for alpha in (1.0, 1e-3):
            eps = 1e-7
            sigma = alpha / (alpha * math.sqrt(min(s, l)) + eps)
            expect = _quintic(sigma, COEFFS, 5) * q
            assert _rel(om.newton_schulz(alpha * q, 5, COEFFS, eps), expect) < 1e-13


def test_ns_equivariances():
    rng = np.random.default_rng(3)
    m = rng.standard_normal((6, 11))
    o = om.newton_schulz(m, 5, COEFFS, 0.0)
    assert _rel(om.newton_schulz(m.T, 5, COEFFS, 0.0), o.T) < 1e-13
    for alpha in (1e3, 1e-4):
        assert _rel(om.newton_schulz(alpha * m, 5, COEFFS, 0.0), o) < 1e-13
    p, _ = np.linalg.qr(rng.standard_normal((6, 6)))
    q, _ = np.linalg.qr(rng.standard_normal((11, 11)))
    assert _rel(om.newton_schulz(p @ m @ q, 5, COEFFS, 0.0), p @ o @ q) < 1e-12


def test_ns_zero_steps_is_normalised_input():
    m = np.arange(12.0).reshape(3, 4)
    assert _rel(om.newton_schulz(m, 0, COEFFS, 0.0), m / np.linalg.norm(m)) < 1e-15


# --- momentum, norms, hyperball ---------------------------------------------

def test_momentum_small_integers():
    m = np.zeros((2, 3))
    seq = []
    for _ in range(3):
        m = om.momentum(m, np.ones((2, 3)), 0.5)
        seq.append(m[0, 0])
    assert seq == [1.0, 1.5, 1.75]


def _r0_pin_holds(capture) -> bool:
    """r0 of a 3-4-12 matrix is exactly 13, and of a random 5 x 7 matrix it
    is the correctly rounded square root of the exact (math.fsum) sum of
    squares, to 1 ulp of float64."""
    w = np.array([[3.0, -4.0], [12.0, 0.0]], np.float32)
    if capture([w])[0] != 13.0:
        return False
    rng = np.random.default_rng(4)
    v = rng.standard_normal((5, 7)).astype(np.float32)
    brute = math.sqrt(math.fsum(float(x) * float(x) for x in v.ravel()))
    return abs(capture([v])[0] - brute) <= 1e-15 * brute


def test_capture_norms_brute_force():
    assert _r0_pin_holds(om.capture_norms)


PLANTED_NORMS = {
    "l1": lambda x: float(np.sum(np.abs(np.asarray(x, np.float64)))),
    "no_sqrt": lambda x: float(np.sum(np.square(np.asarray(x, np.float64)))),
    "max_abs": lambda x: float(np.max(np.abs(np.asarray(x, np.float64)))),
    "fp32_accumulate": lambda x: float(np.sqrt(np.sum(np.square(np.asarray(x, np.float32)), dtype=np.float32))),
    "first_row": lambda x: float(np.linalg.norm(np.asarray(x, np.float64)[0])),
}


@pytest.mark.parametrize("kind", list(PLANTED_NORMS))
def test_planted_norm_mistakes_are_caught(kind, monkeypatch):
    # the mistake goes into the oracle itself: capture_norms then calls the
    # wrong norm, and the brute-force pin above must reject it
    monkeypatch.setattr(om, "frobenius_norm", PLANTED_NORMS[kind])
    assert not _r0_pin_holds(om.capture_norms)


def test_hyperball_norm_invariant_and_fixed_points():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((8, 5)) * 0.02
    o = rng.standard_normal((8, 5))
    r0 = 0.37
    w_new, st = om.hyperball(w, o, 0.02, r0)
    assert st == 0 and abs(np.linalg.norm(w_new) / r0 - 1) < 1e-14
    r_w = float(np.linalg.norm(w))
    w_same, st = om.hyperball(w, o, 0.0, r_w)
    assert st == 0 and _rel(w_same, w) < 1e-15
    w_same, st = om.hyperball(w, np.zeros_like(o), 0.5, r_w)
    assert st == 0 and _rel(w_same, w) < 1e-15


def test_hyperball_degenerate():
    o = np.ones((3, 3))
    w = 0.5 * o
    w_new, st = om.hyperball(w, o, 0.5, 1.0)
    assert st == om.STATUS_DEGENERATE_NORM and np.array_equal(w_new, w)


def test_step_invariants_and_fixed_points():
    rng = np.random.default_rng(6)
    shapes = [(8, 5), (4, 12), (6, 6)]
    ws = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    gs = [(rng.standard_normal(s) * 1e-3).astype(np.float32) for s in shapes]
    ms = [np.zeros(s, np.float32) for s in shapes]
    r0 = om.capture_norms(ws)
    out = om.muonh_step(ws, gs, ms, r0, 0.02, 0.95, 5, COEFFS, 1e-7)
    for w, r, m, g, st in zip(out["w"], r0, out["m"], gs, out["status"]):
        assert st == 0
        assert abs(np.linalg.norm(w.astype(np.float64)) / r - 1) < 1e-6
        assert np.array_equal(m, g)
    zero = om.muonh_step(ws, [np.zeros_like(g) for g in gs], ms, r0, 0.02, 0.95, 5, COEFFS, 1e-7)
    for w_new, w in zip(zero["w"], ws):
        assert np.max(np.abs(w_new - w)) <= 1e-6 * np.max(np.abs(w))
    no_lr = om.muonh_step(ws, gs, ms, r0, 0.0, 0.95, 5, COEFFS, 1e-7)
    for w_new, w in zip(no_lr["w"], ws):
        assert np.max(np.abs(w_new - w)) <= 1e-6 * np.max(np.abs(w))


def test_step_nonfinite_gradient_keeps_weight():
    w = np.full((3, 4), 0.1, np.float32)
    g = np.zeros((3, 4), np.float32)
    g[1, 2] = np.nan
    out = om.muonh_step([w], [g], [np.zeros_like(w)], [1.0], 0.02, 0.95, 5, COEFFS, 1e-7)
    assert out["status"][0] == om.STATUS_NONFINITE_INPUT
    assert np.array_equal(out["w"][0], w)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(4096).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4096),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.0e38, -3.0e38, 1e-40, np.inf, -np.inf],
                 np.float32),
    ]).astype(np.float32)
    # exact ties: low 16 bits == 0x8000, with even and odd kept parts
    ties = (np.arange(64, dtype=np.uint32) << 16 | 0x3F800000 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = om.bf16_round(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# --- golden regression (written by tests/golden/make_golden.py from the oracle) --

def test_golden_small_step_reproduces():
    with open(os.path.join(GOLDEN, "step_small.json")) as f:
        gold = json.load(f)
    p = gold["params"]
    ws = [np.array(c["w"], np.float32) for c in gold["cases"]]
    gs = [np.array(c["g"], np.float32) for c in gold["cases"]]
    ms = [np.array(c["m"], np.float32) for c in gold["cases"]]
    r0 = om.capture_norms(ws)
    out = om.muonh_step(ws, gs, ms, r0, p["lr"], p["beta"], p["ns_steps"], p["coeffs"], p["eps"])
    for case, w, o in zip(gold["cases"], out["w"], out["o"]):
        assert np.array_equal(w, np.array(case["w_new"], np.float32))
        assert np.allclose(o, np.array(case["o"]), rtol=0, atol=1e-14)


# --- planted mistakes: each must be caught by a pin above ---------------------

def _ns_variant(kind):
    def ns(m, steps, coeffs, eps):
        a, b, c = coeffs
        if kind == "swap_bc":
            b, c = c, b
        x = np.array(m, np.float64)
        t = x.shape[0] > x.shape[1]
        if t:
            x = x.T
        x = x / (np.linalg.norm(x) + eps)
        for _ in range(steps):
            g = x @ x.T
            if kind == "drop_cubic":
                p = c * (g @ g)
            elif kind == "sign":
                p = b * g - c * (g @ g)
            else:
                p = b * g + c * (g @ g)
            square = x.shape[0] == x.shape[1]
            x = a * x + (x @ p if kind == "wrong_side" and square else p @ x)
        return x.T if t else x
    return ns


@pytest.mark.parametrize("kind", ["swap_bc", "drop_cubic", "sign", "wrong_side"])
def test_planted_ns_mistakes_are_caught(kind):
    with np.errstate(all="ignore"):
        err = _ns_svd_error(_ns_variant(kind))
    assert not err <= 1e-3
