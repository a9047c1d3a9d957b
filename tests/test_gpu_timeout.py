"""Failure detection on the GPU, without a fault or a hang.

Every pipeline wait of the Newton-Schulz GEMM kernels gives up after a time
limit: the kernel then sets MUONH_STATUS_KERNEL_TIMEOUT, waits (bounded) for
the copies and MMAs it already issued, frees its TMEM and returns, so the
context stays usable.  The test hook muonh_test_gemm_timeout launches one
Gram GEMM whose TMA producer issues nothing and whose waits are limited to
1 ms: the MMA issuer's first wait runs out with nothing in flight.  The
status word must report the timeout, the launch must end within a fraction
of a second, and an ordinary orthogonalisation on the same stream afterwards
must still match the oracle.
"""

import ctypes
import time

import numpy as np
import pytest
import torch

import muonh_workloads as wl
from oracle import muonh as om

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hyperball_constrained_muon_muonh_b300 as mh
    from hyperball_constrained_muon_muonh_b300 import _lib


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mh.get_status()
    yield


@pytest.mark.parametrize("kernel", ["pair", "1sm"])
def test_gemm_wait_times_out_and_context_stays_usable(kernel):
    flags = {"pair": 0, "1sm": _lib.FLAG_GEMM_1SM}[kernel]
    ws = torch.empty(_lib.TEST_TIMEOUT_WS_BYTES, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert mh.get_status() == 0
    t0 = time.perf_counter()
    rc = _lib.lib.muonh_test_gemm_timeout(flags, 1_000_000, ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream)
    assert rc == 0, _lib.lib.muonh_last_error()
    st = mh.get_status()             # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert st & mh.STATUS_KERNEL_TIMEOUT
    assert st & ~mh.STATUS_KERNEL_TIMEOUT == 0
    assert elapsed < 1.0, f"{elapsed:.3f} s: the 1 ms limit did not apply"
    assert mh.get_status() == 0      # reading cleared it

    # the same stream and context still run the real kernels correctly
    g = wl.ragged([(384, 640)]).grad(0, 0, "cuda")
    o = mh.orthogonalize(g, 5, wl.NS_COEFFS, 1e-7, flags=flags)
    want = om.newton_schulz(g.cpu().numpy(), 5, wl.NS_COEFFS, 1e-7)
    got = o.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 3e-2
    assert mh.get_status() == 0
