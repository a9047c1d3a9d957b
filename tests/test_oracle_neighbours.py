"""Pins for the oracle's neighbours of the MuonH step: plain Muon (the
baseline of the Puro-2B paper's matched-ladder comparison, part 6, section
4.3.1) and AdamW (the optimizer of the parameters outside the MuonH group,
model card section "Training").

Muon is pinned by exact rational arithmetic on 1x1 matrices, by its fixed
points and pure-decay case, and by its relation to MuonH (MuonH is Muon
without decay followed by the hyperball retraction).  AdamW is pinned by
torch.optim.AdamW run in float64 (an independent library implementation of
the textbook method) and by its closed-form first step.  Planted mistakes
(flipped sign, coupled decay, missing bias correction...) must each fail a
pin.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import muonh as om

COEFFS = (3.4445, -4.7750, 2.0315)


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------------------
# Muon
# ---------------------------------------------------------------------------

def _muon_scalar_exact(w, g, lr, beta, wd, steps=5, eps=1e-7):
    """One Muon step on a 1x1 matrix (momentum starting at 0) in exact rationals."""
    m = Fraction(g)                     # beta * 0 + g
    x = m / (abs(m) + Fraction(eps))
    a, b, c = (Fraction(v) for v in COEFFS)
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return (1 - Fraction(lr) * Fraction(wd)) * Fraction(w) - Fraction(lr) * x


def _muon_scalar_case(update):
    """Largest relative error of `update` (in place of om.muon_update) on 1x1 cases."""
    worst = 0.0
    orig = om.muon_update
    om.muon_update = update
    try:
        for w, g, lr, wd in ((0.3, 0.75, 0.02, 0.1), (-1.5, -3.0, 0.5, 0.0), (2.0, 1e-3, 0.1, 0.25)):
            out = om.muon_step([np.array([[w]])], [np.array([[g]])], [np.zeros((1, 1))], lr, 0.95, wd, 5,
                               COEFFS, 1e-7, state_dtype=None)
            want = float(_muon_scalar_exact(w, g, lr, 0.95, wd))
            worst = max(worst, abs(out["w"][0][0, 0] - want) / abs(want))
    finally:
        om.muon_update = orig
    return worst


def test_muon_scalar_exact_rational():
    assert _muon_scalar_case(om.muon_update) <= 4e-16


@pytest.mark.parametrize("kind", ["sign", "coupled_decay", "decay_after"])
def test_planted_muon_mistakes_are_caught(kind):
    bad = {
        "sign": lambda w, o, lr, wd: (1 - lr * wd) * np.asarray(w, np.float64) + lr * np.asarray(o, np.float64),
        "coupled_decay": lambda w, o, lr, wd: (1 + lr * wd) * np.asarray(w, np.float64) - lr * np.asarray(o, np.float64),
        "decay_after": lambda w, o, lr, wd: (1 - lr * wd) * (np.asarray(w, np.float64) - lr * np.asarray(o, np.float64)),
    }[kind]
    assert _muon_scalar_case(bad) > 1e-6


def test_muon_fixed_points_and_pure_decay():
    rng = np.random.default_rng(7)
    w = [rng.standard_normal((6, 9)).astype(np.float32), rng.standard_normal((9, 6)).astype(np.float32)]
    z = [np.zeros_like(x) for x in w]
    g = [rng.standard_normal(x.shape).astype(np.float32) for x in w]
    # zero gradient and momentum: O = NS(0) = 0, so W only decays
    for wd in (0.0, 0.1):
        out = om.muon_step(w, z, z, 0.02, 0.95, wd, 5, COEFFS, 1e-7, state_dtype=None)
        for a, b in zip(out["w"], w):
            assert np.array_equal(a, (1 - 0.02 * wd) * b.astype(np.float64))
    # zero learning rate: nothing moves
    out = om.muon_step(w, g, z, 0.0, 0.95, 0.1, 5, COEFFS, 1e-7, state_dtype=None)
    for a, b in zip(out["w"], w):
        assert np.array_equal(a, b.astype(np.float64))


def test_muonh_is_undecayed_muon_retracted():
    rng = np.random.default_rng(8)
    w = [rng.standard_normal((5, 12)), rng.standard_normal((12, 5))]
    g = [rng.standard_normal(x.shape) for x in w]
    m = [rng.standard_normal(x.shape) for x in w]
    r0 = om.capture_norms(w)
    mu = om.muon_step(w, g, m, 0.05, 0.9, 0.0, 5, COEFFS, 1e-7, state_dtype=None)
    mh = om.muonh_step(w, g, m, r0, 0.05, 0.9, 5, COEFFS, 1e-7, state_dtype=None)
    for u, got, radius in zip(mu["w"], mh["w"], r0):
        assert _rel(got, radius * u / np.linalg.norm(u)) < 1e-14


def test_muon_nonfinite_gradient_keeps_weight():
    w = [np.ones((3, 4), np.float32)]
    g = [np.full((3, 4), np.nan, np.float32)]
    out = om.muon_step(w, g, [np.zeros((3, 4), np.float32)], 0.02, 0.95, 0.1, 5, COEFFS, 1e-7)
    assert out["status"][0] == om.STATUS_NONFINITE_INPUT
    assert np.array_equal(out["w"][0], w[0])


# ---------------------------------------------------------------------------
# AdamW
# ---------------------------------------------------------------------------

def _torch_adamw(params, grads_per_step, lr, betas, eps, wd):
    ps = [torch.tensor(p, dtype=torch.float64, requires_grad=True) for p in params]
    opt = torch.optim.AdamW(ps, lr=lr, betas=betas, eps=eps, weight_decay=wd, foreach=False)
    hist = []
    for grads in grads_per_step:
        for p, g in zip(ps, grads):
            p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        hist.append([p.detach().numpy().copy() for p in ps])
    return hist


def _oracle_adamw(params, grads_per_step, lr, betas, eps, wd, step_fn=None):
    step_fn = step_fn or om.adamw_step
    p = [np.asarray(x, np.float64) for x in params]
    m = [np.zeros_like(x) for x in p]
    v = [np.zeros_like(x) for x in p]
    hist = []
    for t, grads in enumerate(grads_per_step, start=1):
        out = step_fn(p, grads, m, v, t, lr, betas[0], betas[1], eps, wd, state_dtype=None)
        p, m, v = out["p"], out["m"], out["v"]
        hist.append([x.copy() for x in p])
    return hist


def _adamw_case(seed=11):
    rng = np.random.default_rng(seed)
    params = [rng.standard_normal(s) for s in ((7,), (3, 5), (2, 3, 4))]
    grads = [[rng.standard_normal(p.shape) * 1e-2 for p in params] for _ in range(4)]
    return params, grads


def _adamw_worst(step_fn=None):
    params, grads = _adamw_case()
    cfg = dict(lr=1e-2, betas=(0.9, 0.95), eps=1e-8, wd=0.1)
    ref = _torch_adamw(params, grads, **cfg)
    got = _oracle_adamw(params, grads, step_fn=step_fn, **cfg)
    return max(_rel(a, b) for ha, hb in zip(got, ref) for a, b in zip(ha, hb))


def test_adamw_matches_torch_float64():
    assert _adamw_worst() < 1e-13


def test_adamw_first_step_closed_form():
    # from zero moments, m_hat = g and v_hat = g^2 at step 1
    rng = np.random.default_rng(12)
    p = rng.standard_normal((4, 6))
    g = rng.standard_normal((4, 6))
    lr, wd, eps = 3e-3, 0.1, 1e-8
    out = om.adamw_step([p], [g], [np.zeros_like(p)], [np.zeros_like(p)], 1, lr, 0.9, 0.95, eps, wd,
                        state_dtype=None)
    want = (1 - lr * wd) * p - lr * g / (np.abs(g) + eps)
    assert _rel(out["p"][0], want) < 1e-15


@pytest.mark.parametrize("kind", ["no_bias_correction", "coupled_decay", "eps_inside_sqrt", "beta_swap"])
def test_planted_adamw_mistakes_are_caught(kind):
    def bad(params, grads, ms, vs, step, lr, b1, b2, eps, wd, state_dtype=None):
        out = {"p": [], "m": [], "v": []}
        for p, g, m, v in zip(params, grads, ms, vs):
            if kind == "coupled_decay":
                g = g + wd * p
            if kind == "beta_swap":
                b1, b2 = b2, b1
            m = b1 * m + (1 - b1) * g
            v = b2 * v + (1 - b2) * g * g
            mh, vh = (m, v) if kind == "no_bias_correction" else (m / (1 - b1 ** step), v / (1 - b2 ** step))
            den = np.sqrt(vh + eps) if kind == "eps_inside_sqrt" else np.sqrt(vh) + eps
            decay = 1.0 if kind == "coupled_decay" else (1 - lr * wd)
            out["p"].append(decay * p - lr * mh / den)
            out["m"].append(m)
            out["v"].append(v)
        return out
    assert _adamw_worst(bad) > 1e-9


# ---------------------------------------------------------------------------
# Nesterov momentum and update scales (variants offered as flags)
# ---------------------------------------------------------------------------

def test_nesterov_input_small_integers():
    # beta = 0.5, G = 1 every step: M = 1, 1.5, 1.75; look-ahead X = G + beta*M = 1.5, 1.75, 1.875
    m = np.zeros((1, 1))
    g = np.ones((1, 1))
    for want_m, want_x in ((1.0, 1.5), (1.5, 1.75), (1.75, 1.875)):
        m = om.momentum(m, g, 0.5)
        assert m[0, 0] == want_m
        assert om.ns_input(m, g, 0.5, True)[0, 0] == want_x
        assert om.ns_input(m, g, 0.5, False)[0, 0] == want_m


def test_nesterov_with_zero_beta_is_heavy_ball():
    rng = np.random.default_rng(21)
    w = [rng.standard_normal((6, 10))]
    g = [rng.standard_normal((6, 10))]
    m = [rng.standard_normal((6, 10))]
    r0 = om.capture_norms(w)
    a = om.muonh_step(w, g, m, r0, 0.02, 0.0, 5, COEFFS, 1e-7, state_dtype=None, nesterov=True)
    b = om.muonh_step(w, g, m, r0, 0.02, 0.0, 5, COEFFS, 1e-7, state_dtype=None, nesterov=False)
    assert np.array_equal(a["w"][0], b["w"][0])


def test_nesterov_changes_the_step():
    rng = np.random.default_rng(22)
    w, g, m = (rng.standard_normal((6, 10)) for _ in range(3))
    a = om.muon_step([w], [g], [m], 0.02, 0.9, 0.0, 5, COEFFS, 1e-7, state_dtype=None, nesterov=True)
    want = om.muon_update(w, om.newton_schulz(g + 0.9 * (0.9 * m + g), 5, COEFFS, 1e-7), 0.02, 0.0)
    assert _rel(a["w"][0], want) < 1e-14


def test_update_scale_values():
    assert om.update_scale(4, 4, "shape") == 1.0
    assert om.update_scale(8, 2, "shape") == 2.0          # tall: sqrt(8/2)
    assert om.update_scale(2, 8, "shape") == 1.0          # wide: max(1, 2/8)
    assert om.update_scale(8, 2, "rms") == 0.2 * math.sqrt(8)
    assert om.update_scale(2, 8, "rms") == 0.2 * math.sqrt(8)
    assert om.update_scale(5, 3, "none") == 1.0


@pytest.mark.parametrize("kind", ["shape", "rms"])
def test_scaled_step_is_step_with_scaled_rate(kind):
    # U = W - lr*(s*O) is the unscaled step at rate lr*s
    rng = np.random.default_rng(23)
    for shape in ((8, 2), (2, 8), (5, 5)):
        w, g = rng.standard_normal(shape), rng.standard_normal(shape)
        z = np.zeros(shape)
        sc = om.update_scale(*shape, kind)
        r0 = om.capture_norms([w])
        a = om.muonh_step([w], [g], [z], r0, 0.02, 0.9, 5, COEFFS, 1e-7, state_dtype=None, scale=kind)
        b = om.muonh_step([w], [g], [z], r0, 0.02 * sc, 0.9, 5, COEFFS, 1e-7, state_dtype=None)
        assert _rel(a["w"][0], b["w"][0]) < 1e-14
        c = om.muon_step([w], [g], [z], 0.02, 0.9, 0.1, 5, COEFFS, 1e-7, state_dtype=None, scale=kind)
        o = om.newton_schulz(g, 5, COEFFS, 1e-7)
        assert _rel(c["w"][0], (1 - 0.02 * 0.1) * w - 0.02 * sc * o) < 1e-14
