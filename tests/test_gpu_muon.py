"""GPU parity of plain Muon (muon_step, the baseline MuonH is compared with)
against the float64 oracle, through the C ABI.

Tolerance: the Newton-Schulz output O carries a relative Frobenius error of
at most 3e-2 with bf16 tensor-core operands (1e-4 in the fp32 check mode);
W_new = (1 - lr*wd)*W - lr*O moves by lr*err(O), so
    ||W_gpu - W_oracle|| <= lr * tol_O * ||O|| + 1e-6 * ||W_oracle||
(the last term: fp32 rounding of the stored weight).  The momentum must be
within 2 ulp, and the bf16 weight copy must be the RNE rounding of the
kernel's own fp32 weight, bit for bit.
"""

import numpy as np
import pytest
import torch

import muonh_workloads as wl
from oracle import muonh as om

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh

TOL_O = {False: 3e-2, True: 1e-4}
MODES = {"pair": 0, "one_step": 1 << 8, "1sm": 1 << 3, "fp32": 1}
RAGGED = [(300, 200), (200, 300), (13, 37), (37, 13), (77, 77), (520, 129), (8, 1), (1, 1), (640, 384)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield
    assert mh.get_status() & mh.STATUS_KERNEL_TIMEOUT == 0


def _f32(x):
    return float(np.float32(x))


def _run_and_check(work, steps, wd, mode="pair", idx=None):
    fp32 = mode == "fp32"
    idx = list(range(len(work.shapes))) if idx is None else idx
    ws = work.weights("cuda")
    opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=wd, ns_steps=work.ns_steps, ns_coeffs=work.coeffs,
                  eps=work.eps, bf16_copies=True, flags=MODES[mode])
    lr, beta, eps = _f32(work.lr), _f32(work.beta), _f32(work.eps)
    coeffs = tuple(_f32(c) for c in work.coeffs)
    tol = TOL_O[fp32]
    for t in range(steps):
        gs = work.grads(t, "cuda")
        w_prev = [ws[i].cpu().numpy() for i in idx]
        m_prev = [opt.moms[i].cpu().numpy() for i in idx]
        opt.step(gs)
        torch.cuda.synchronize()
        out = om.muon_step(w_prev, [gs[i].cpu().numpy() for i in idx], m_prev, lr, beta, _f32(wd), work.ns_steps,
                           coeffs, eps)
        for k, i in enumerate(idx):
            m_or = out["m"][k]
            ulp = np.spacing(np.abs(m_or).astype(np.float32))
            assert np.all(np.abs(opt.moms[i].cpu().numpy() - m_or) <= 2 * ulp), f"momentum of matrix {i}"
            w = ws[i].cpu().numpy().astype(np.float64)
            w_or = out["w"][k].astype(np.float64)
            o = out["o"][k]
            bound = lr * tol * np.linalg.norm(o) + 1e-6 * np.linalg.norm(w_or)
            err = np.linalg.norm(w - w_or)
            assert err <= bound, f"step {t} matrix {i} {work.shapes[i]}: {err:.3e} > {bound:.3e}"
            want_b = om.bf16_round(ws[i].cpu().numpy())
            got_b = opt.bf16[i].float().cpu().numpy()
            assert np.array_equal(got_b.view(np.uint32), want_b.view(np.uint32))
    assert mh.get_status() == 0


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_muon_ragged_shapes(mode, wd):
    _run_and_check(wl.ragged(RAGGED), 2, wd, mode)


@pytest.mark.parametrize("ns_steps", [0, 1, 2])
def test_muon_short_iteration_counts(ns_steps):
    work = wl.ragged(RAGGED)
    work.ns_steps = ns_steps
    _run_and_check(work, 2, 0.1)


@pytest.mark.parametrize("mode", ["pair", "1sm"])
def test_muon_qwen3_layer(mode):
    _run_and_check(wl.qwen3_layer(), 2, 0.1, mode)


def test_muon_aspect_low_rank():
    _run_and_check(wl.aspect_16384x1024(), 1, 0.1, "pair")


def test_muonh_is_undecayed_muon_retracted_on_gpu():
    # same momentum and Newton-Schulz: MuonH's W is r0 * U / ||U|| with U the
    # weight plain Muon (no decay) writes, to fp32 rounding
    work = wl.ragged([(256, 384), (384, 256), (77, 77)])
    wa, wb = work.weights("cuda"), work.weights("cuda")
    a = mh.Muon(wa, lr=work.lr, beta=work.beta, weight_decay=0.0)
    b = mh.MuonH(wb, lr=work.lr, beta=work.beta)
    gs = work.grads(0, "cuda")
    a.step(gs)
    b.step(gs)
    for u, w, r0 in zip(wa, wb, b.r0):
        want = (r0.double() * u.double() / u.double().norm()).cpu()
        assert torch.allclose(w.double().cpu(), want, rtol=0, atol=4e-7 * want.abs().max().item())
    assert mh.get_status() == 0


def test_muon_nonfinite_gradient_keeps_weight():
    work = wl.ragged([(64, 32), (32, 64)])
    ws = work.weights("cuda")
    keep = [w.clone() for w in ws]
    opt = mh.Muon(ws, weight_decay=0.1)
    gs = work.grads(0, "cuda")
    gs[1][2, 3] = float("inf")
    opt.step(gs)
    assert mh.get_status() & mh.STATUS_NONFINITE_INPUT
    assert torch.equal(ws[1], keep[1])
    assert not torch.equal(ws[0], keep[0])


def test_muon_deterministic_bitwise():
    work = wl.ragged([(512, 384), (384, 512), (77, 77)])
    outs = []
    for _ in range(2):
        ws = work.weights("cuda")
        opt = mh.Muon(ws, weight_decay=0.1, bf16_copies=True)
        for t in range(2):
            opt.step(work.grads(t, "cuda"))
        outs.append([w.clone() for w in ws] + [m.clone() for m in opt.moms])
    for x, y in zip(*outs):
        assert torch.equal(x, y)
