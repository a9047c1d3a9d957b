"""GPU parity of AdamW (adamw_step, the optimizer of the parameters outside
the MuonH group) against the float64 oracle, through the C ABI.

Tolerances, from the fp32 arithmetic of one element:
  * m = fma(beta1, m0, (1-beta1)*g): two roundings, each at most an ulp of
    the terms, which may nearly cancel, so
    |m_gpu - m_oracle| <= 2^-22 * (|beta1*m0| + |(1-beta1)*g|);
  * v = fma(beta2, v0, (1-beta2)*g*g): three roundings of positive terms, so
    within 4 ulp of the result (1e-30 absolute near zero);
  * p: p*decay (one rounding) plus step_size * m / (sqrt(v)*c + eps) (about
    eight roundings), plus the error of m carried through m_hat / denom:
    |p_gpu - p_oracle| <= 2^-20 * (|p| + lr*|u|) + lr * dm / ((1-beta1^t) * denom)
    with u = m_hat / (sqrt(v_hat) + eps) and denom = sqrt(v_hat) + eps from
    the oracle and dm the bound on m above;
  * the bf16 copy is the RNE rounding of the kernel's own fp32 p, bit for bit.
"""

import numpy as np
import pytest
import torch

import muonh_workloads as wl
from oracle import muonh as om

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh

SHAPES = [(1,), (3,), (4,), (5, 7), (1000,), (4097,), (65536 + 5,), (2, 3, 4), (300, 200), (131072,)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield


def _f32(x):
    return float(np.float32(x))


def _ulp_ok(got, want, k=4):
    want32 = np.asarray(want, np.float32)
    tol = k * np.spacing(np.abs(want32)) + 1e-30
    return np.all(np.abs(np.asarray(got, np.float64) - want32.astype(np.float64)) <= tol)


def _check(params, grads_fn, steps, lr, betas, eps, wd):
    opt = mh.AdamW(params, lr=lr, betas=betas, eps=eps, weight_decay=wd, bf16_copies=True)
    lr32, b1, b2, e32, wd32 = _f32(lr), _f32(betas[0]), _f32(betas[1]), _f32(eps), _f32(wd)
    for t in range(1, steps + 1):
        gs = grads_fn(t)
        p0 = [p.cpu().numpy() for p in params]
        m0 = [m.cpu().numpy() for m in opt.exp_avgs]
        v0 = [v.cpu().numpy() for v in opt.exp_avg_sqs]
        opt.step(gs)
        torch.cuda.synchronize()
        out = om.adamw_step(p0, [g.cpu().numpy() for g in gs], m0, v0, t, lr32, b1, b2, e32, wd32, state_dtype=None)
        for i in range(len(params)):
            g64 = gs[i].cpu().numpy().astype(np.float64)
            dm = 2.0 ** -22 * (np.abs(b1 * m0[i].astype(np.float64)) + np.abs((1 - b1) * g64)) + 1e-30
            got_m = opt.exp_avgs[i].cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got_m - out["m"][i]) <= dm), f"m of tensor {i} at step {t}"
            assert _ulp_ok(opt.exp_avg_sqs[i].cpu().numpy(), out["v"][i]), f"v of tensor {i} at step {t}"
            m_hat = out["m"][i] / (1 - b1 ** t)
            v_hat = out["v"][i] / (1 - b2 ** t)
            denom = np.sqrt(v_hat) + e32
            u = m_hat / denom
            tol = 2.0 ** -20 * (np.abs(out["p"][i]) + lr32 * np.abs(u)) + lr32 * dm / ((1 - b1 ** t) * denom)
            got = params[i].cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got - out["p"][i]) <= tol), f"p of tensor {i} at step {t}"
            want_b = om.bf16_round(params[i].cpu().numpy())
            assert np.array_equal(opt.bf16[i].float().cpu().numpy().view(np.uint32), want_b.view(np.uint32))


def _rand(shape, seed, scale, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * scale


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_adamw_ragged_tensors(wd):
    params = [_rand(s, 100 + i, 0.02) for i, s in enumerate(SHAPES)]
    _check(params, lambda t: [_rand(s, 1000 * t + i, 1e-2) for i, s in enumerate(SHAPES)], 3, 2e-3, (0.9, 0.95),
           1e-8, wd)


def test_adamw_zero_and_sparse_gradients():
    # zero gradients keep v at 0 (denominator eps); mixed magnitudes span the exponent range
    params = [_rand(s, 200 + i, 1.0) for i, s in enumerate(SHAPES[:6])]

    def grads(t):
        out = []
        for i, s in enumerate(SHAPES[:6]):
            g = _rand(s, 3000 * t + i, 1.0)
            g = g * torch.pow(10.0, _rand(s, 5000 * t + i, 3.0).round())
            g[g.abs() < 1e-2] = 0.0
            out.append(g)
        return out
    _check(params, grads, 3, 1e-3, (0.8, 0.99), 1e-8, 0.1)


def test_adamw_group_sample():
    # the AdamW group's embedding and a few norm vectors
    work = wl.adamw_group()
    idx = [0, 1, 2, 60, 112]
    params = [work.weight(i, "cuda").reshape(-1) for i in idx]
    _check(params, lambda t: [work.grad(i, t, "cuda").reshape(-1) for i in idx], 2, work.lr, (0.9, 0.95), 1e-8,
           0.1)


def test_adamw_many_tensors():
    # more tensors than one descriptor batch carries
    shapes = [(17,), (64,), (129,)] * 250
    params = [_rand(s, 7 + i, 0.1) for i, s in enumerate(shapes)]
    _check(params, lambda t: [_rand(s, 100000 * t + i, 1e-2) for i, s in enumerate(shapes)], 1, 1e-3, (0.9, 0.95),
           1e-8, 0.1)
