"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle.

Tolerances (from the MuonH step's arithmetic and the stated targets):
  * Newton-Schulz output O: relative Frobenius error <= 3e-2 with bf16
    tensor-core operands, <= 1e-4 in the fp32 check mode;
  * momentum: fp32 fma against the float64 value rounded to fp32, <= 2 ulp;
  * | ||W||_F / r0 - 1 | <= 1e-5;
  * new W: an error eps_O in O moves U = W - lr*O by lr*eps_O*||O||, so
    rel_err(W) <= 2*lr*tol_O*||O||/||U|| + 1e-6 (fp32 rounding);
  * the bf16 weight copy equals round-to-nearest-even of the kernel's own
    fp32 weight, bit for bit (both sides round the same fp32 values).
"""

import math

import numpy as np
import pytest
import torch

import muonh_workloads as wl
from oracle import muonh as om

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh

TOL_O = {0: 3e-2, 1: 1e-4}   # keyed by fp32_check


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield
    assert mh.get_status() & mh.STATUS_KERNEL_TIMEOUT == 0


def _run_steps(work, steps=1, fp32_check=False, device="cuda", indices=None, bf16=True, flags=0):
    """GPU MuonH over `work`; returns host copies of inputs and outputs per step."""
    idx = list(range(len(work.shapes))) if indices is None else indices
    ws = work.weights(device)
    w0 = [ws[i].cpu().numpy() for i in idx]
    opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs,
                   eps=work.eps, bf16_copies=bf16, fp32_check=fp32_check, flags=flags)
    r0 = opt.r0.cpu().numpy()
    hist = []
    for t in range(steps):
        gs = work.grads(t, device)
        m_prev = [opt.moms[i].cpu().numpy() for i in idx]
        w_prev = [ws[i].cpu().numpy() for i in idx]
        opt.step(gs)
        torch.cuda.synchronize()
        hist.append({
            "g": [gs[i].cpu().numpy() for i in idx],
            "m_prev": m_prev, "w_prev": w_prev,
            "w": [ws[i].cpu().numpy() for i in idx],
            "m": [opt.moms[i].cpu().numpy() for i in idx],
            "wb": [opt.bf16[i].float().cpu().numpy() for i in idx] if bf16 else None,
        })
        del gs
    status = mh.get_status()
    return w0, r0[idx], hist, status


def _f32(x):
    """The value the library receives for a float argument."""
    return float(np.float32(x))


def _check_step(work, w0, r0_gpu, hist, fp32_check, idx=None):
    idx = list(range(len(work.shapes))) if idx is None else idx
    lr, beta, eps = _f32(work.lr), _f32(work.beta), _f32(work.eps)
    coeffs = tuple(_f32(c) for c in work.coeffs)
    # r0 against the oracle's norm of the initial weights
    r0_or = om.capture_norms(w0)
    assert np.max(np.abs(r0_gpu / r0_or - 1)) < 1e-6
    tol = TOL_O[int(fp32_check)]
    for h in hist:
        out = om.muonh_step(h["w_prev"], h["g"], h["m_prev"], r0_gpu.astype(np.float64), lr,
                            beta, work.ns_steps, coeffs, eps)
        for k in range(len(idx)):
            m_or = out["m"][k]
            ulp = np.spacing(np.abs(m_or).astype(np.float32))
            assert np.all(np.abs(h["m"][k] - m_or) <= 2 * ulp), f"momentum of matrix {idx[k]}"
            w = h["w"][k].astype(np.float64)
            assert abs(np.linalg.norm(w) / r0_gpu[k] - 1) <= 1e-5, f"norm of matrix {idx[k]}"
            o = out["o"][k]
            u = h["w_prev"][k].astype(np.float64) - lr * o
            bound = 2 * lr * tol * np.linalg.norm(o) / np.linalg.norm(u) + 1e-6
            err = _rel(w, out["w"][k])
            assert err <= bound, f"W of matrix {idx[k]}: {err:.3e} > {bound:.3e}"
            if h["wb"] is not None:
                want = om.bf16_round(h["w"][k])
                assert np.array_equal(h["wb"][k].view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------------------
# Newton-Schulz alone (muonh_orthogonalize) against the oracle
# ---------------------------------------------------------------------------

NS_SHAPES = [(256, 128), (128, 256), (300, 200), (200, 300), (129, 520), (520, 129), (1, 1), (1, 8), (8, 1),
             (77, 77), (640, 384), (2048, 2048), (1024, 2048), (6144, 2048), (2048, 6144)]


# flag sets: the default 2-SM pair GEMM, the 1-SM GEMM, the fp32 check mode
MODES = {"pair": 0, "one_step": 1 << 8, "1sm": 1 << 3, "fp32": 1}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("shape", NS_SHAPES)
def test_orthogonalize_matches_oracle(shape, mode):
    fp32_check = int(mode == "fp32")
    work = wl.ragged([shape])
    g = work.grad(0, 0, "cuda")
    o = mh.orthogonalize(g, 5, wl.NS_COEFFS, 1e-7, flags=MODES[mode])
    torch.cuda.synchronize()
    want = om.newton_schulz(g.cpu().numpy(), 5, wl.NS_COEFFS, 1e-7)
    err = _rel(o.cpu().numpy(), want)
    assert err <= TOL_O[fp32_check], f"{shape}: {err:.3e}"
    assert mh.get_status() == 0


@pytest.mark.parametrize("mode", ["pair", "1sm", "fp32"])
@pytest.mark.parametrize("shape", [(300, 200), (200, 300), (2048, 1024), (1024, 2048), (256, 128), (64, 32),
                                   (129, 520)])
def test_orthogonalize_bf16_input_and_output(shape, mode):
    # bf16 in: widened exactly, so the result equals the fp32 call on the
    # widened values bit for bit; bf16 out: the round-to-nearest-even of the
    # fp32 result, bit for bit; both against the oracle within the Newton-
    # Schulz tolerance (plus bf16 rounding of O, <= 2^-9 relative per element)
    flags = MODES[mode]
    g = wl.ragged([shape]).grad(0, 0, "cuda")
    x16 = g.to(torch.bfloat16)
    xw = x16.float()
    o32 = mh.orthogonalize(xw, 5, wl.NS_COEFFS, 1e-7, flags=flags)
    o_in16 = mh.orthogonalize(x16, 5, wl.NS_COEFFS, 1e-7, flags=flags)
    o_out16 = mh.orthogonalize(xw, 5, wl.NS_COEFFS, 1e-7, flags=flags, out_dtype=torch.bfloat16)
    o_both16 = mh.orthogonalize(x16, 5, wl.NS_COEFFS, 1e-7, flags=flags, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert o_in16.dtype == torch.float32 and o_out16.dtype == torch.bfloat16
    assert torch.equal(o_in16, o32)
    assert torch.equal(o_both16, o_out16)
    want_bits = om.bf16_round(o32.cpu().numpy()).view(np.uint32) >> 16
    assert np.array_equal(o_out16.cpu().view(torch.int16).numpy().view(np.uint16).astype(np.uint32), want_bits)
    want = om.newton_schulz(xw.cpu().numpy(), 5, wl.NS_COEFFS, 1e-7)
    tol = TOL_O[int(mode == "fp32")]
    assert _rel(o32.cpu().numpy(), want) <= tol
    assert _rel(o_out16.float().cpu().numpy(), want) <= tol + 4e-3
    assert mh.get_status() == 0


@pytest.mark.parametrize("shape", [(16384, 1024), (1024, 16384), (1024, 2048), (4096, 1024), (1024, 3000),
                                   (65536, 256)])
def test_split_k_gram_repeatable(shape):
    # alone, these matrices' Grams have at most 16 pair tiles, so K is split
    # into ranges (2 to 8 here, the last one shorter where K is ragged) whose
    # partial products are summed in range order by whichever range finishes
    # last: repeated calls agree bit for bit, and with the oracle within the
    # tolerance
    g = wl.ragged([shape]).grad(0, 0, "cuda")
    outs = [mh.orthogonalize(g, 5, wl.NS_COEFFS, 1e-7) for _ in range(3)]
    torch.cuda.synchronize()
    assert mh.get_status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    want = om.newton_schulz(g.cpu().numpy(), 5, wl.NS_COEFFS, 1e-7)
    assert _rel(outs[0].cpu().numpy(), want) <= TOL_O[0]


@pytest.mark.parametrize("steps", [0, 1, 2])
def test_orthogonalize_step_counts(steps):
    g = wl.ragged([(384, 640)]).grad(0, 0, "cuda")
    for fp32 in (0, 1):
        o = mh.orthogonalize(g, steps, wl.NS_COEFFS, 1e-7, flags=mh.FLAG_FP32_CHECK if fp32 else 0)
        want = om.newton_schulz(g.cpu().numpy(), steps, wl.NS_COEFFS, 1e-7)
        assert _rel(o.cpu().numpy(), want) <= TOL_O[fp32]


def test_orthogonalize_low_rank_aspect():
    # rank-8 input: the fp32 Newton-Schulz state keeps the null directions clean
    work = wl.aspect_16384x1024()
    for i in (0, 4):
        g = work.grad(i, 0, "cuda")
        want = om.newton_schulz(g.cpu().numpy(), 5, wl.NS_COEFFS, 1e-7)
        for flags in (0, MODES["1sm"]):
            o = mh.orthogonalize(g, 5, wl.NS_COEFFS, 1e-7, flags=flags)
            assert _rel(o.cpu().numpy(), want) <= TOL_O[0]


# ---------------------------------------------------------------------------
# full MuonH step against the oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fp32_check", [False, True])
def test_step_single_256x128(fp32_check):
    work = wl.single_256x128()
    w0, r0, hist, status = _run_steps(work, 1, fp32_check)
    assert status == 0
    _check_step(work, w0, r0, hist, fp32_check)


@pytest.mark.parametrize("mode", list(MODES))
def test_step_ragged_shapes_three_steps(mode):
    fp32_check = mode == "fp32"
    work = wl.ragged([(300, 200), (200, 300), (129, 520), (1, 8), (8, 1), (77, 77), (5, 3), (1, 1), (640, 384)])
    w0, r0, hist, status = _run_steps(work, 3, fp32_check, flags=MODES[mode])
    assert status == 0
    _check_step(work, w0, r0, hist, fp32_check)


@pytest.mark.parametrize("mode", ["pair", "1sm"])
@pytest.mark.parametrize("ns_steps", [0, 1, 2])
def test_step_short_iteration_counts(ns_steps, mode):
    # one iteration: the same apply launch reads X from the momentum and
    # writes U = W - lr*O; zero iterations: O is the normalised momentum
    work = wl.ragged([(300, 200), (200, 300), (13, 37), (37, 13), (77, 77), (520, 129), (8, 1)])
    work.ns_steps = ns_steps
    w0, r0, hist, status = _run_steps(work, 2, False, flags=MODES[mode])
    assert status == 0
    _check_step(work, w0, r0, hist, False)


@pytest.mark.parametrize("mode", list(MODES))
def test_step_qwen3_layer(mode):
    fp32_check = mode == "fp32"
    work = wl.qwen3_layer()
    w0, r0, hist, status = _run_steps(work, 2, fp32_check, flags=MODES[mode])
    assert status == 0
    _check_step(work, w0, r0, hist, fp32_check)


def test_step_batched_256_heavy_tails():
    work = wl.batched_256()
    idx = list(range(0, 1024, 73))
    w0, r0, hist, status = _run_steps(work, 1, False, indices=idx)
    assert status == 0
    _check_step(work, w0, r0, hist, False, idx=idx)


def test_step_aspect_low_rank():
    work = wl.aspect_16384x1024()
    idx = [0, 5]
    w0, r0, hist, status = _run_steps(work, 1, False, indices=idx)
    assert status == 0
    _check_step(work, w0, r0, hist, False, idx=idx)


@pytest.mark.parametrize("mode", ["pair", "one_stream"])
def test_step_maximum_side_lengths(mode):
    # the longest side the ABI accepts (MUONH_MAX_SIDE = 65536), tall and wide,
    # with a short side on fp32 CUDA cores (8) and on the tensor cores (96:
    # one ragged pair tile, 1024 K steps in the Gram)
    work = wl.ragged([(65536, 8), (8, 65536), (65536, 96), (96, 65536)])
    flags = {"pair": 0, "one_stream": mh.FLAG_ONE_STREAM}[mode]
    w0, r0, hist, status = _run_steps(work, 2, False, flags=flags)
    assert status == 0
    _check_step(work, w0, r0, hist, False)


def test_step_golden_fixture():
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "step_small.json")) as f:
        gold = json.load(f)
    p = gold["params"]
    ws = [torch.tensor(c["w"], dtype=torch.float32, device="cuda") for c in gold["cases"]]
    gs = [torch.tensor(c["g"], dtype=torch.float32, device="cuda") for c in gold["cases"]]
    for flags in (0, mh.FLAG_FP32_CHECK):
        wcur = [w.clone() for w in ws]
        opt = mh.MuonH(wcur, lr=p["lr"], beta=p["beta"], ns_steps=p["ns_steps"], ns_coeffs=p["coeffs"],
                       eps=p["eps"], fp32_check=bool(flags))
        for m, c in zip(opt.moms, gold["cases"]):
            m.copy_(torch.tensor(c["m"], dtype=torch.float32))
        opt.step(gs)
        tol = TOL_O[int(bool(flags))]
        for w, c in zip(wcur, gold["cases"]):
            o = np.array(c["o"])
            u = np.array(c["w"], np.float64) - p["lr"] * o
            bound = 2 * p["lr"] * tol * np.linalg.norm(o) / np.linalg.norm(u) + 1e-6
            assert _rel(w.cpu().numpy(), np.array(c["w_new"])) <= bound
    assert mh.get_status() == 0


# ---------------------------------------------------------------------------
# degenerate cases, status word, determinism, resume
# ---------------------------------------------------------------------------

def test_nonfinite_gradient_keeps_weight_and_sets_status():
    work = wl.ragged([(64, 32), (32, 64)])
    ws = work.weights("cuda")
    keep = [w.clone() for w in ws]
    opt = mh.MuonH(ws)
    gs = work.grads(0, "cuda")
    gs[0][3, 5] = float("nan")
    opt.step(gs)
    st = mh.get_status()
    assert st & mh.STATUS_NONFINITE_INPUT
    assert torch.equal(ws[0], keep[0])
    assert not torch.equal(ws[1], keep[1])           # the other matrix still moves
    assert abs(ws[1].double().norm().item() / opt.r0[1].item() - 1) < 1e-5


# shapes that take each path of the step: the fused tensor-core path (row
# length a multiple of 4), the unfused one (hyperball norm pass), the on-chip
# small-matrix kernel, fp32 CUDA cores for short sides <= 80, and the fp32
# check mode
DEGENERATE_PATHS = {"pair": ((384, 512), 0), "unfused": ((300, 202), 0), "small": ((256, 128), 0),
                    "cuda_cores": ((64, 32), 0), "fp32": ((384, 512), 1)}


@pytest.mark.parametrize("case", ["zero_lr", "zero_grad"])
@pytest.mark.parametrize("path", list(DEGENERATE_PATHS))
def test_degenerate_norm_sets_status(path, case):
    # W = 0 (so r0 = 0) stepped with lr = 0, or with G = 0 (then M = 0 and
    # O = 0): U = W - lr*O is exactly zero in any arithmetic, so ||U|| = 0,
    # the status bit is set and W is kept.  A second matrix of the same
    # shape with ordinary inputs is stepped in the same call.
    shape, fp32 = DEGENERATE_PATHS[path]
    work = wl.ragged([shape, shape])
    ws = work.weights("cuda")
    ws[0].zero_()
    keep = [w.clone() for w in ws]
    lr = 0.0 if case == "zero_lr" else 0.02
    opt = mh.MuonH(ws, lr=lr, fp32_check=bool(fp32), bf16_copies=True)
    assert opt.r0[0].item() == 0.0
    gs = work.grads(0, "cuda")
    if case == "zero_grad":
        gs[0].zero_()
    opt.step(gs)
    st = mh.get_status()
    assert st == mh.STATUS_DEGENERATE_NORM
    assert torch.equal(ws[0], keep[0])                    # kept: still all zero
    assert torch.equal(opt.moms[0], gs[0])                # the momentum still moves (M = beta*0 + G)
    assert abs(ws[1].double().norm().item() / opt.r0[1].item() - 1) < 1e-5
    if case == "zero_grad":
        assert not torch.equal(ws[1], keep[1])            # the ordinary matrix moves


def test_zero_gradient_and_zero_lr_fixed_points():
    work = wl.ragged([(96, 64), (64, 96)])
    for lr, zero_grad in ((0.02, True), (0.0, False)):
        ws = work.weights("cuda")
        keep = [w.clone() for w in ws]
        opt = mh.MuonH(ws, lr=lr)
        gs = [torch.zeros_like(w) for w in ws] if zero_grad else work.grads(0, "cuda")
        opt.step(gs)
        for w, k in zip(ws, keep):
            assert torch.allclose(w, k, rtol=0, atol=2e-6 * k.abs().max().item())
    assert mh.get_status() == 0


def test_deterministic_bitwise():
    work = wl.ragged([(512, 384), (384, 512), (256, 256)])
    outs = []
    for _ in range(2):
        ws = work.weights("cuda")
        opt = mh.MuonH(ws, bf16_copies=True)
        for t in range(2):
            opt.step(work.grads(t, "cuda"))
        outs.append([w.clone() for w in ws] + [m.clone() for m in opt.moms])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_resume_matches_uninterrupted():
    work = wl.ragged([(256, 384), (384, 256)])
    ws_a = work.weights("cuda")
    a = mh.MuonH(ws_a)
    for t in range(4):
        a.step(work.grads(t, "cuda"))
    ws_b = work.weights("cuda")
    b = mh.MuonH(ws_b)
    for t in range(2):
        b.step(work.grads(t, "cuda"))
    sd = b.state_dict()
    saved_w = [w.clone() for w in ws_b]
    ws_c = [w.clone() for w in saved_w]
    c = mh.MuonH(ws_c)
    c.load_state_dict(sd)
    for t in range(2, 4):
        c.step(work.grads(t, "cuda"))
    for x, y in zip(ws_a, ws_c):
        assert torch.equal(x, y)


def test_capture_norms_many_matrices():
    work = wl.ragged([(3, 5), (1, 1), (4097, 3), (1000, 1000)] * 150)   # > one descriptor batch
    ws = work.weights("cuda")
    r0 = mh.capture_norms(ws).cpu().numpy()
    want = om.capture_norms([w.cpu().numpy() for w in ws])
    assert np.max(np.abs(r0 / want - 1)) < 1e-6


def test_many_matrices_step():
    # more matrices than one descriptor batch carries
    work = wl.ragged([(32, 48), (48, 32), (16, 16)] * 200)
    idx = [0, 1, 2, 301, 599]
    w0, r0, hist, status = _run_steps(work, 1, False, indices=idx)
    assert status == 0
    _check_step(work, w0, r0, hist, False, idx=idx)


def _sharded_world1(rank, port, result):
    import os
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        import hyperball_constrained_muon_muonh_b300 as mh_
        work = wl.ragged([(256, 384), (384, 256), (512, 512), (96, 100)])
        wa, wb = work.weights("cuda"), work.weights("cuda")
        a = mh_.ShardedMuonH(wa, lr=work.lr, beta=work.beta)
        b = mh_.MuonH(wb, lr=work.lr, beta=work.beta)
        for t in range(2):
            gs = work.grads(t, "cuda")
            a.step(gs)
            b.step(gs)
        torch.cuda.synchronize()
        result[0] = int(all(torch.equal(x, y) for x, y in zip(wa, wb)) and set(a.owners) == {0})
    finally:
        dist.destroy_process_group()


def test_sharded_world_size_1_equals_unsharded():
    # one rank owns every matrix: the sharded step is the plain step, bit for bit
    # (several ranks on one GPU would wait on one another; the exchange across
    # ranks is tested with gloo on CPU)
    import socket
    import torch.multiprocessing as tmp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = tmp.get_context("spawn")
    result = ctx.Manager().dict()
    tmp.start_processes(_sharded_world1, args=(port, result), nprocs=1, start_method="spawn", join=True)
    assert result.get(0) == 1
