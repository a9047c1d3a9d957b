"""GPU parity of the small-matrix path: matrices with both sides <= 256 (and
a short side above 80) take the whole step -- momentum, every Newton-Schulz
iteration, the hyperball or Muon update -- in one kernel per CTA pair with
the iterations on chip.  Checked against the float64 oracle through the C ABI
with the tolerances of the other parity tests (MuonH: ||W||/r0 within 1e-5 and
rel_err(W) <= 2*lr*tol*||O||/||U|| + 1e-6; Muon: ||dW|| <= lr*tol*||O|| +
1e-6*||W||; tol = 3e-2 for bf16 tensor-core operands), momentum within 2 ulp,
and the bf16 copy bit-exact to the kernel's own fp32 weight.
"""

import numpy as np
import pytest
import torch

import muonh_workloads as wl
from oracle import muonh as om

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh

# wide, tall (transposed on load and store), square, ragged; row lengths of
# 0, 4 (mod 8) and odd, so every vector and scalar path of the kernel runs
SHAPES = [(256, 256), (256, 128), (128, 256), (100, 250), (250, 100), (96, 96), (200, 256), (129, 97),
          (100, 196), (96, 100)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield
    assert mh.get_status() & mh.STATUS_KERNEL_TIMEOUT == 0


def _f32(x):
    return float(np.float32(x))


def _run(work, optimizer, steps=2, flags=0, nesterov=False, scale="none", wd=0.1, idx=None):
    ws = work.weights("cuda")
    idx = list(range(len(ws))) if idx is None else idx
    if optimizer == "muonh":
        opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs, eps=work.eps,
                       bf16_copies=True, flags=flags)
        r0 = opt.r0.cpu().numpy().astype(np.float64)
    else:
        opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=wd, ns_steps=work.ns_steps,
                      ns_coeffs=work.coeffs, eps=work.eps, bf16_copies=True, flags=flags)
    lr, beta, eps = _f32(work.lr), _f32(work.beta), _f32(work.eps)
    coeffs = tuple(_f32(c) for c in work.coeffs)
    for t in range(steps):
        gs = work.grads(t, "cuda")
        w0 = [ws[i].cpu().numpy() for i in idx]
        m0 = [opt.moms[i].cpu().numpy() for i in idx]
        opt.step(gs)
        torch.cuda.synchronize()
        g0 = [gs[i].cpu().numpy() for i in idx]
        if optimizer == "muonh":
            out = om.muonh_step(w0, g0, m0, r0[idx], lr, beta, work.ns_steps, coeffs, eps, nesterov=nesterov,
                                scale=scale)
        else:
            out = om.muon_step(w0, g0, m0, lr, beta, _f32(wd), work.ns_steps, coeffs, eps, nesterov=nesterov,
                               scale=scale)
        for k, i in enumerate(idx):
            m_or = out["m"][k]
            assert np.all(np.abs(opt.moms[i].cpu().numpy() - m_or) <= 2 * np.spacing(np.abs(m_or).astype(np.float32))), \
                f"momentum of matrix {i}"
            w = ws[i].cpu().numpy().astype(np.float64)
            o = out["o"][k]
            if optimizer == "muonh":
                assert abs(np.linalg.norm(w) / r0[i] - 1) <= 1e-5, f"norm of matrix {i}"
                u = w0[k].astype(np.float64) - lr * o
                bound = 2 * lr * 3e-2 * np.linalg.norm(o) / np.linalg.norm(u) + 1e-6
                err = np.linalg.norm(w - out["w"][k]) / np.linalg.norm(out["w"][k])
            else:
                bound = lr * 3e-2 * np.linalg.norm(o) + 1e-6 * np.linalg.norm(out["w"][k])
                err = np.linalg.norm(w - out["w"][k])
            assert err <= bound, f"{optimizer} step {t} matrix {i} {work.shapes[i]}: {err:.3e} > {bound:.3e}"
            want_b = om.bf16_round(ws[i].cpu().numpy())
            assert np.array_equal(opt.bf16[i].float().cpu().numpy().view(np.uint32), want_b.view(np.uint32))
    assert mh.get_status() == 0
    return opt


@pytest.mark.parametrize("optimizer", ["muonh", "muon"])
def test_small_shapes(optimizer):
    opt = _run(wl.ragged(SHAPES), optimizer)
    assert opt is not None


def test_small_kernel_is_the_path_taken():
    # the step's profile shows the small-matrix kernel and no Newton-Schulz GEMM launches
    work = wl.ragged([(256, 256), (128, 256)])
    ws = work.weights("cuda")
    opt = mh.MuonH(ws)
    mh.lib.muonh_profile_enable(1)
    opt.step(work.grads(0, "cuda"))
    prof = mh.profile_read()
    mh.lib.muonh_profile_enable(0)
    assert "small_step" in prof
    assert not any(k.startswith("ns_") for k in prof)


@pytest.mark.parametrize("steps_ns", [1, 2])
def test_small_short_iteration_counts(steps_ns):
    work = wl.ragged(SHAPES)
    work.ns_steps = steps_ns
    _run(work, "muonh")


def test_small_variants():
    _run(wl.ragged(SHAPES), "muonh", flags=mh.FLAG_NESTEROV | mh.FLAG_SCALE_SHAPE, nesterov=True, scale="shape")
    _run(wl.ragged(SHAPES), "muon", flags=mh.FLAG_SCALE_RMS, scale="rms")


@pytest.mark.parametrize("g_scale,eps", [(1e12, 1e-7), (1e-12, 0.0)])
def test_small_extreme_norms_fold_the_scale_into_x(g_scale, eps):
    # The kernel keeps X in TMEM up to a scalar sigma (starting at
    # 1/(||M|| + eps), times a per iteration).  Gradients of 1e12 (sigma below
    # 2^-32) and of 1e-12 with eps = 0 (sigma above 2^32) make it fold sigma
    # into X instead, at the first iteration; the result must not change.
    work = wl.ragged(SHAPES[:6])
    work.g_scale, work.eps = g_scale, eps
    _run(work, "muonh")
    _run(work, "muon")


@pytest.mark.parametrize("coeffs", [(0.0, 1.5, -0.5), (1.5, -0.5, 0.0)])
def test_small_coefficients_with_a_zero_term(coeffs):
    # a = 0: no a*X term (the scale cannot be kept in sigma); c = 0: no A*A product
    work = wl.ragged(SHAPES[:6])
    work.coeffs = coeffs
    _run(work, "muonh")
    _run(work, "muon")


def test_small_batched_more_than_one_launch():
    # 1024 matrices of 256 x 256 (the batched workload) need two launches
    work = wl.batched_256()
    _run(work, "muonh", steps=1, idx=list(range(0, 1024, 97)) + [1023])


def test_small_single_256x128_golden_workload():
    _run(wl.single_256x128(), "muonh", steps=3)


def test_small_nonfinite_keeps_weight():
    work = wl.ragged([(128, 128), (96, 112)])
    ws = work.weights("cuda")
    keep = [w.clone() for w in ws]
    opt = mh.MuonH(ws)
    gs = work.grads(0, "cuda")
    gs[0][5, 7] = float("nan")
    opt.step(gs)
    assert mh.get_status() & mh.STATUS_NONFINITE_INPUT
    assert torch.equal(ws[0], keep[0])
    assert abs(ws[1].double().norm().item() / opt.r0[1].item() - 1) < 1e-5


def test_small_deterministic_bitwise():
    work = wl.ragged([(256, 256), (250, 100), (96, 96)])
    outs = []
    for _ in range(2):
        ws = work.weights("cuda")
        opt = mh.MuonH(ws, bf16_copies=True)
        for t in range(2):
            opt.step(work.grads(t, "cuda"))
        outs.append([w.clone() for w in ws] + [m.clone() for m in opt.moms])
    for x, y in zip(*outs):
        assert torch.equal(x, y)
