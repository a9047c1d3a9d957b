"""GPU parity of the step variants offered as flags (Nesterov momentum and
the update scales) for MuonH and plain Muon, against the float64 oracle run
with the matching parameters, through the C ABI.

Tolerances as in the parity tests of the plain steps:
  * MuonH: ||W||/r0 within 1e-5, rel_err(W) <= 2*lr*tol_O*||O||/||U|| + 1e-6;
  * Muon: ||W_gpu - W_oracle|| <= lr*tol_O*||O|| + 1e-6*||W_oracle||;
with O the oracle's scaled update and tol_O = 3e-2 (bf16 tensor cores) or
1e-4 (fp32 check mode); momentum within 2 ulp.
"""

import numpy as np
import pytest
import torch

import muonh_workloads as wl
from oracle import muonh as om

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh

SHAPES = [(300, 200), (200, 300), (13, 37), (37, 13), (77, 77), (520, 129), (640, 384), (8, 1)]
NEST, SHAPE, RMS = 0x2, 0x10, 0x20
VARIANTS = {"nesterov": (NEST, True, "none"), "shape": (SHAPE, False, "shape"), "rms": (RMS, False, "rms"),
            "nesterov+shape": (NEST | SHAPE, True, "shape"), "nesterov+rms": (NEST | RMS, True, "rms")}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield
    assert mh.get_status() & mh.STATUS_KERNEL_TIMEOUT == 0


def _f32(x):
    return float(np.float32(x))


def _run(work, optimizer, flags, nesterov, scale, steps=2, wd=0.1, extra=0):
    fp32 = bool(extra & mh.FLAG_FP32_CHECK)
    tol = 1e-4 if fp32 else 3e-2
    ws = work.weights("cuda")
    if optimizer == "muonh":
        opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, flags=flags | extra)
        r0 = opt.r0.cpu().numpy().astype(np.float64)
    else:
        opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=wd, ns_steps=work.ns_steps, flags=flags | extra)
    lr, beta, eps = _f32(work.lr), _f32(work.beta), _f32(work.eps)
    coeffs = tuple(_f32(c) for c in work.coeffs)
    for t in range(steps):
        gs = work.grads(t, "cuda")
        w0 = [w.cpu().numpy() for w in ws]
        m0 = [m.cpu().numpy() for m in opt.moms]
        opt.step(gs)
        torch.cuda.synchronize()
        g0 = [g.cpu().numpy() for g in gs]
        if optimizer == "muonh":
            out = om.muonh_step(w0, g0, m0, r0, lr, beta, work.ns_steps, coeffs, eps, nesterov=nesterov, scale=scale)
        else:
            out = om.muon_step(w0, g0, m0, lr, beta, _f32(wd), work.ns_steps, coeffs, eps, nesterov=nesterov,
                               scale=scale)
        for i in range(len(ws)):
            m_or = out["m"][i]
            assert np.all(np.abs(opt.moms[i].cpu().numpy() - m_or) <= 2 * np.spacing(np.abs(m_or).astype(np.float32)))
            w = ws[i].cpu().numpy().astype(np.float64)
            o = out["o"][i]
            if optimizer == "muonh":
                assert abs(np.linalg.norm(w) / r0[i] - 1) <= 1e-5
                u = w0[i].astype(np.float64) - lr * o
                bound = 2 * lr * tol * np.linalg.norm(o) / np.linalg.norm(u) + 1e-6
                err = np.linalg.norm(w - out["w"][i]) / np.linalg.norm(out["w"][i])
            else:
                bound = lr * tol * np.linalg.norm(o) + 1e-6 * np.linalg.norm(out["w"][i])
                err = np.linalg.norm(w - out["w"][i])
            assert err <= bound, f"{optimizer} step {t} matrix {i} {work.shapes[i]}: {err:.3e} > {bound:.3e}"
    assert mh.get_status() == 0


@pytest.mark.parametrize("optimizer", ["muonh", "muon"])
@pytest.mark.parametrize("variant", list(VARIANTS))
def test_variants_ragged(optimizer, variant):
    flags, nest, scale = VARIANTS[variant]
    _run(wl.ragged(SHAPES), optimizer, flags, nest, scale)


@pytest.mark.parametrize("extra", [0x8, 0x1])
def test_variants_other_gemm_modes(extra):
    flags, nest, scale = VARIANTS["nesterov+shape"]
    _run(wl.ragged(SHAPES), "muonh", flags, nest, scale, extra=extra)


def test_variants_qwen3_layer():
    flags, nest, scale = VARIANTS["nesterov+shape"]
    _run(wl.qwen3_layer(), "muonh", flags, nest, scale)
    flags, nest, scale = VARIANTS["rms"]
    _run(wl.qwen3_layer(), "muon", flags, nest, scale)


def test_variants_zero_iterations():
    work = wl.ragged(SHAPES)
    work.ns_steps = 0
    for opt in ("muonh", "muon"):
        flags, nest, scale = VARIANTS["nesterov+shape"]
        _run(work, opt, flags, nest, scale)


def test_scale_flags_exclude_each_other():
    w = [torch.zeros(8, 8, device="cuda") + 0.1]
    with pytest.raises(mh.MuonHError):
        opt = mh.MuonH(w, flags=SHAPE | RMS)
        opt.step([torch.ones(8, 8, device="cuda")])


@pytest.mark.parametrize("optimizer", ["muonh", "muon"])
def test_bf16_gradients(optimizer):
    # gradients handed over as bf16 (MUONH_FLAG_GRAD_BF16); the oracle gets the same values widened
    work = wl.ragged(SHAPES + [(256, 256), (250, 100)])
    ws = work.weights("cuda")
    flags = 0x40
    if optimizer == "muonh":
        opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, flags=flags)
        r0 = opt.r0.cpu().numpy().astype(np.float64)
    else:
        opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=0.1, flags=flags)
    lr, beta, eps = _f32(work.lr), _f32(work.beta), _f32(work.eps)
    coeffs = tuple(_f32(c) for c in work.coeffs)
    for t in range(2):
        gb = [g.to(torch.bfloat16) for g in work.grads(t, "cuda")]
        w0 = [w.cpu().numpy() for w in ws]
        m0 = [m.cpu().numpy() for m in opt.moms]
        opt.step(gb)
        torch.cuda.synchronize()
        g0 = [g.float().cpu().numpy() for g in gb]
        if optimizer == "muonh":
            out = om.muonh_step(w0, g0, m0, r0, lr, beta, work.ns_steps, coeffs, eps)
        else:
            out = om.muon_step(w0, g0, m0, lr, beta, _f32(0.1), work.ns_steps, coeffs, eps)
        for i in range(len(ws)):
            m_or = out["m"][i]
            assert np.all(np.abs(opt.moms[i].cpu().numpy() - m_or) <= 2 * np.spacing(np.abs(m_or).astype(np.float32)))
            w = ws[i].cpu().numpy().astype(np.float64)
            o = out["o"][i]
            if optimizer == "muonh":
                u = w0[i].astype(np.float64) - lr * o
                bound = 2 * lr * 3e-2 * np.linalg.norm(o) / np.linalg.norm(u) + 1e-6
                err = np.linalg.norm(w - out["w"][i]) / np.linalg.norm(out["w"][i])
            else:
                bound = lr * 3e-2 * np.linalg.norm(o) + 1e-6 * np.linalg.norm(out["w"][i])
                err = np.linalg.norm(w - out["w"][i])
            assert err <= bound, f"{optimizer} step {t} matrix {i}: {err:.3e} > {bound:.3e}"
    assert mh.get_status() == 0
