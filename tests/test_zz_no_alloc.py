"""muonh_orthogonalize_static: Newton-Schulz for callers that cannot allocate.

Some callers cannot call cudaMalloc at all: code running inside an allocator
or memory-pool callback, processes held to a fixed device-memory budget, or
hosts that must not grow their device footprint after start-up.  For them the
library offers one entry point whose scratch is a fixed array in the
library's own device memory instead of a caller-supplied workspace.  These
tests call it through the C ABI and hold it to the workspace entry point
(muonh_orthogonalize) on the same inputs, for calls in a row: both run the
same deterministic kernels, so the results must agree bit for bit, and a call
that read stale scratch from the previous one would show up.

This file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

import muonh_workloads as wl
from hyperball_constrained_muon_muonh_b300 import _lib

COEFFS = (ctypes.c_float * 3)(*wl.NS_COEFFS)


def _static(x, out, flags):
    return _lib.lib.muonh_orthogonalize_static(
        ctypes.c_void_p(x.data_ptr()), _lib.DTYPE_F32, ctypes.c_void_p(out.data_ptr()), _lib.DTYPE_F32, x.shape[0],
        x.shape[1], 5, COEFFS, 1e-7, flags, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _with_workspace(x, flags):
    need = ctypes.c_size_t()
    assert _lib.lib.muonh_orthogonalize_workspace_size(x.shape[0], x.shape[1], flags, ctypes.byref(need)) == 0
    ws = torch.empty(need.value, dtype=torch.uint8, device=x.device)
    out = torch.empty_like(x)
    rc = _lib.lib.muonh_orthogonalize(
        ctypes.c_void_p(x.data_ptr()), _lib.DTYPE_F32, ctypes.c_void_p(out.data_ptr()), _lib.DTYPE_F32, x.shape[0],
        x.shape[1], 5, COEFFS, 1e-7, flags, ctypes.c_void_p(ws.data_ptr()), need.value,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, _lib.lib.muonh_last_error()
    return out


def test_static_rejects_oversized_shapes():
    # checked on the host before any device work
    x = ctypes.c_void_p(256)
    rc = _lib.lib.muonh_orthogonalize_static(x, _lib.DTYPE_F32, x, _lib.DTYPE_F32, 4096, 4096, 5, COEFFS, 1e-7, 0,
                                             None)
    assert rc == _lib.ERR_WORKSPACE
    assert b"96 MiB" in _lib.lib.muonh_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("flags", [0, _lib.FLAG_FP32_CHECK])
def test_static_matches_workspace_entry_two_calls(flags):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # two calls in a row with different shapes (one ragged, one tall), then the
    # first shape again: each result must equal the workspace entry point's
    cases = [wl.ragged([(300, 200)]).grad(0, 0, "cuda"),
             wl.ragged([(2048, 1024)]).grad(0, 1, "cuda"),
             wl.ragged([(300, 200)]).grad(0, 2, "cuda")]
    for x in cases:
        out = torch.full_like(x, float("nan"))
        rc = _static(x, out, flags)
        assert rc == 0, _lib.lib.muonh_last_error()
        ref = _with_workspace(x, flags)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref)
    st = ctypes.c_uint32()
    assert _lib.lib.muonh_get_status(ctypes.byref(st), None) == 0
    assert st.value == 0
