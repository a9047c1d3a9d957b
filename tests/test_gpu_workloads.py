"""GPU parity at the full sizes of the benchmark workloads, several steps.

The step runs on every matrix of the workload, in the launch configuration
bench.py times (the default pair GEMM, buckets of up to 56 same-shape
matrices spread over the side streams); the float64 oracle then re-runs the
same steps on a sample of the matrices, which is exact per matrix because
matrices are independent.  Each step's sample is checked and dropped before
the next one (host memory stays at a few GB):
  * the 2B set (28 Qwen3-style decoder layers, 196 matrices): ten
    consecutive steps with fresh gradients, layers 0 and 27 (all seven
    shapes, the first and last matrix of every bucket);
  * 1024 independent 256 x 256 matrices with Student-t3 gradients: three
    steps, every matrix;
  * four 16384 x 1024 and four 1024 x 16384 matrices with rank-8 gradients:
    three steps, every matrix.
Tolerances are those of test_gpu_parity.py: O within 3e-2 (bf16 tensor-core
operands), momentum within 2 ulp, | ||W||/r0 - 1 | <= 1e-5, the derived
bound on W, and the bf16 weight copy bit-exact.
"""

import numpy as np
import pytest
import torch

import muonh_workloads as wl
from oracle import muonh as om

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh

TOL_O = 3e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield
    torch.cuda.empty_cache()


def _f32(x):
    return float(np.float32(x))


def _host(ts, idx):
    return [ts[i].cpu().numpy() for i in idx]


def _run_and_check(work, steps, idx):
    ws = work.weights("cuda")
    opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs, eps=work.eps,
                   bf16_copies=True)
    r0 = opt.r0.cpu().numpy()[idx].astype(np.float64)
    w0 = _host(ws, idx)
    assert np.max(np.abs(r0 / om.capture_norms(w0) - 1)) < 1e-6
    lr, beta, eps = _f32(work.lr), _f32(work.beta), _f32(work.eps)
    coeffs = tuple(_f32(c) for c in work.coeffs)
    for t in range(steps):
        gs = work.grads(t, "cuda")
        w_prev, m_prev, g = _host(ws, idx), _host(opt.moms, idx), _host(gs, idx)
        opt.step(gs)
        del gs
        w_new, m_new = _host(ws, idx), _host(opt.moms, idx)
        wb = [opt.bf16[i].float().cpu().numpy() for i in idx]
        assert mh.get_status() == 0, f"step {t}"
        out = om.muonh_step(w_prev, g, m_prev, r0, lr, beta, work.ns_steps, coeffs, eps)
        for k, i in enumerate(idx):
            where = f"step {t}, matrix {i} {work.shapes[i]}"
            ulp = np.spacing(np.abs(out["m"][k]).astype(np.float32))
            assert np.all(np.abs(m_new[k] - out["m"][k]) <= 2 * ulp), f"momentum, {where}"
            w = w_new[k].astype(np.float64)
            assert abs(np.linalg.norm(w) / r0[k] - 1) <= 1e-5, f"norm, {where}"
            o = out["o"][k]
            u = w_prev[k].astype(np.float64) - lr * o
            bound = 2 * lr * TOL_O * np.linalg.norm(o) / np.linalg.norm(u) + 1e-6
            err = np.linalg.norm(w - out["w"][k]) / np.linalg.norm(out["w"][k])
            assert err <= bound, f"W, {where}: {err:.3e} > {bound:.3e}"
            assert np.array_equal(wb[k].view(np.uint32), om.bf16_round(w_new[k]).view(np.uint32)), f"bf16, {where}"
        del w_prev, m_prev, g, w_new, m_new, wb, out


def test_qwen3_2b_ten_steps_layers_0_and_27():
    work = wl.qwen3_2b()
    assert len(work.shapes) == 196
    idx = list(range(0, 7)) + list(range(27 * 7, 28 * 7))
    _run_and_check(work, 10, idx)


def test_batched_1024x256x256_three_steps_every_matrix():
    work = wl.batched_256()
    _run_and_check(work, 3, list(range(1024)))


def test_aspect_16384x1024_three_steps_every_matrix():
    work = wl.aspect_16384x1024()
    _run_and_check(work, 3, list(range(8)))
