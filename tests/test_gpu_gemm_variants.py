"""Newton-Schulz GEMM variants against the default CTA-pair kernel, bit for
bit.

The default pair kernel stages two 64-wide K steps per pipeline stage (one
32 KB TMA box per operand) when K and the contiguous extent of every
MN-major operand are multiples of 64, else one.  MUONH_FLAG_GEMM_ONE_STEP
forces one K step per stage (16 KB boxes); MUONH_FLAG_ONE_STREAM keeps every launch on the caller's stream
instead of spreading independent buckets over side streams (same kernels,
same dependencies).  All GEMM kernels walk the same list of 256 x 256 pair tiles and issue
the same tcgen05 MMAs on the same shared-memory layout in the same K order,
so every output -- O, the momentum, W, the bf16 copy -- must be identical.
The shapes cover: symmetric Gram/polynomial tile lists with even and odd
counts, the wide apply (tiles that share B; B is MN-major), the tall
apply and tall Gram (A shared; the tall Gram's operands are MN-major), an
odd number of K steps, consecutive tiles that straddle a row, a column or a
matrix boundary, buckets of several matrices, and shapes that fall back to
one K step (K or an MN-major extent not a multiple of 64).  The oracle
parity of each variant runs in test_gpu_parity.py and test_gpu_muon.py.
"""

import numpy as np
import pytest
import torch

import muonh_workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield
    assert mh.get_status() & mh.STATUS_KERNEL_TIMEOUT == 0


# (rows, cols): short side s -> s/256 pair tiles per side
#   2048^2: 36 Gram tiles (even), wide apply 8 x 8
#   640x384: 3 Gram tiles (odd), apply 2 x 3 over a ragged 128-row tail, 5 K steps (odd)
#   768x1280, 1280x768: apply 3 x 5, super-tiles across column / row ends
#   129x520, 520x129: one tile per launch; K = 520, one K step per stage
#   1280x320, 320x1280: MN-major Gram operands and apply B with extents % 64 == 0
#   384x650, 650x384: MN-major extent 650 -> one K step per stage
#   6144x2048, 2048x6144: the tall and wide MLP shapes
SHAPES = [(2048, 2048), (640, 384), (384, 640), (768, 1280), (1280, 768), (129, 520), (520, 129),
          (1280, 320), (320, 1280), (384, 650), (650, 384), (6144, 2048), (2048, 6144), (1000, 1000)]

VARIANTS = ["one_step", "one_stream"]


def _flag(variant):
    return {"one_step": mh.FLAG_GEMM_ONE_STEP,
            "one_stream": mh.FLAG_ONE_STREAM}[variant]


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES)
def test_orthogonalize_variant_equals_pair(shape, variant):
    g = wl.ragged([shape]).grad(0, 0, "cuda")
    o_pair = mh.orthogonalize(g, 5, wl.NS_COEFFS, 1e-7, flags=0)
    o_var = mh.orthogonalize(g, 5, wl.NS_COEFFS, 1e-7, flags=_flag(variant))
    torch.cuda.synchronize()
    assert mh.get_status() == 0
    assert np.array_equal(_bits(o_pair), _bits(o_var)), f"{shape}"


def _step_states(work, steps, flags, optimizer="muonh", wd=0.0):
    ws = work.weights("cuda")
    if optimizer == "muonh":
        opt = mh.MuonH(ws, lr=work.lr, beta=work.beta, ns_steps=work.ns_steps, ns_coeffs=work.coeffs,
                       eps=work.eps, bf16_copies=True, flags=flags)
    else:
        opt = mh.Muon(ws, lr=work.lr, beta=work.beta, weight_decay=wd, ns_steps=work.ns_steps,
                      ns_coeffs=work.coeffs, eps=work.eps, bf16_copies=True, flags=flags)
    for t in range(steps):
        opt.step(work.grads(t, "cuda"))
    torch.cuda.synchronize()
    return ([_bits(w) for w in ws], [_bits(m) for m in opt.moms],
            [opt.bf16[i].detach().cpu().view(torch.int16).numpy() for i in range(len(ws))])


# several matrices per bucket: super-tiles that pair the last tile of one
# matrix with the first of the next
BUCKETS = [(512, 512)] * 3 + [(384, 1024)] * 5 + [(1024, 384)] * 3 + [(2048, 768)] * 2 + [(300, 200), (77, 77)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("optimizer", ["muonh", "muon"])
@pytest.mark.parametrize("extra", [0, 1 << 1])   # plain, Nesterov (the first apply reads its own input)
def test_step_variant_equals_pair(optimizer, extra, variant):
    work = wl.ragged(BUCKETS)
    a = _step_states(work, 2, extra, optimizer, wd=0.1)
    b = _step_states(work, 2, extra | _flag(variant), optimizer, wd=0.1)
    assert mh.get_status() == 0
    for k in range(len(BUCKETS)):
        for part in range(3):
            assert np.array_equal(a[part][k], b[part][k]), f"matrix {k} {BUCKETS[k]} part {part}"


@pytest.mark.parametrize("variant", VARIANTS)
def test_step_variant_equals_pair_qwen3_layer(variant):
    work = wl.qwen3_layer()
    a = _step_states(work, 2, 0)
    b = _step_states(work, 2, _flag(variant))
    assert mh.get_status() == 0
    for k in range(len(work.shapes)):
        for part in range(3):
            assert np.array_equal(a[part][k], b[part][k]), f"matrix {k} part {part}"
