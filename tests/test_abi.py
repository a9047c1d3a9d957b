"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/muonh.h declares, rejects bad arguments before any launch, and sizes
workspaces from shapes alone."""

import ctypes
import os
import re

import pytest

from hyperball_constrained_muon_muonh_b300 import _lib
import hyperball_constrained_muon_muonh_b300 as mh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b((?:muonh|muon|adamw)_[a-z0-9_]+)\s*\(", text))
    return names


def test_header_declarations_are_exported():
    declared = _declared()
    assert declared >= set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(_lib.lib, name), name


def test_binding_constants_match_header():
    # every MUONH_FLAG_* / _STATUS_* / _ERR_* value the header defines is the
    # binding's constant of the same name, and every binding flag is declared
    text = open(os.path.join(ROOT, "include", "muonh.h")).read()
    defs = {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"#define\s+MUONH_((?:FLAG|STATUS|ERR)_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", text)}
    dtypes = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+MUONH_(DTYPE_[A-Z0-9]+)\s+(\d+)", text)}
    assert dtypes == {"DTYPE_F32": _lib.DTYPE_F32, "DTYPE_BF16": _lib.DTYPE_BF16}
    assert len(defs) >= 16   # 4 error codes, 3 status bits, 9 flags
    for name, value in defs.items():
        assert getattr(_lib, name) == value, name
    for name in dir(_lib):
        if name.startswith("FLAG_"):
            assert name in defs, name
    flags = [v for k, v in defs.items() if k.startswith("FLAG_")]
    assert len(set(flags)) == len(flags)                      # distinct bits
    assert all(v and (v & (v - 1)) == 0 for v in flags)       # one bit each


def test_version_and_strings():
    assert _lib.lib.muonh_version() >= 100
    assert _lib.lib.muonh_status_string(0) == b"ok"
    assert _lib.lib.muonh_status_string(2).startswith(b"workspace")


def _arr(shapes, ptr=256):
    arr = (_lib.MatrixT * len(shapes))()
    for i, (r, c) in enumerate(shapes):
        arr[i].rows, arr[i].cols = r, c
        arr[i].w = arr[i].grad = arr[i].mom = ptr
    return arr


COEFFS = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)


def _step(arr, n=None, r0=256, lr=0.02, beta=0.95, steps=5, coeffs=COEFFS, eps=1e-7, flags=0, ws=256,
          ws_bytes=1 << 40):
    return _lib.lib.muonh_step(arr, len(arr) if n is None else n, ctypes.c_void_p(r0), lr, beta, steps, coeffs,
                               eps, flags, ctypes.c_void_p(ws), ws_bytes, None)


def test_step_rejects_bad_arguments_before_launch():
    good = _arr([(4, 4)])
    assert _lib.lib.muonh_step(None, 1, None, 0.02, 0.95, 5, COEFFS, 1e-7, 0, None, 0, None) == _lib.ERR_INVALID_ARG
    assert _step(good, n=0) == _lib.ERR_INVALID_ARG
    assert _step(_arr([(0, 4)])) == _lib.ERR_INVALID_ARG
    assert _step(_arr([(4, 70000)])) == _lib.ERR_INVALID_ARG
    assert _step(_arr([(4, 4)], ptr=260)) == _lib.ERR_INVALID_ARG          # misaligned
    assert _step(good, r0=0) == _lib.ERR_INVALID_ARG
    assert _step(good, lr=float("nan")) == _lib.ERR_INVALID_ARG
    assert _step(good, steps=-1) == _lib.ERR_INVALID_ARG
    assert _step(good, steps=65) == _lib.ERR_INVALID_ARG
    assert _step(good, coeffs=(ctypes.c_float * 3)(1.0, float("inf"), 0.0)) == _lib.ERR_INVALID_ARG
    assert _step(good, eps=-1.0) == _lib.ERR_INVALID_ARG
    assert _step(good, flags=0x400) == _lib.ERR_UNSUPPORTED
    assert _step(good, flags=0x80) == _lib.ERR_UNSUPPORTED     # no flag has this bit
    assert _step(good, ws=0) == _lib.ERR_WORKSPACE
    assert _step(good, ws=512 + 16) == _lib.ERR_WORKSPACE
    assert _step(good, ws_bytes=16) == _lib.ERR_WORKSPACE
    assert b"workspace too small" in _lib.lib.muonh_last_error()
    nullgrad = _arr([(4, 4)])
    nullgrad[0].grad = None
    assert _step(nullgrad) == _lib.ERR_INVALID_ARG


def test_capture_and_orthogonalize_reject_bad_arguments():
    assert _lib.lib.muonh_capture_norms(None, 1, None, None) == _lib.ERR_INVALID_ARG
    assert _lib.lib.muonh_capture_norms(_arr([(4, 4)]), 1, None, None) == _lib.ERR_INVALID_ARG
    o = _lib.lib.muonh_orthogonalize
    p, f32, bf16 = ctypes.c_void_p(256), _lib.DTYPE_F32, _lib.DTYPE_BF16
    assert o(None, f32, None, f32, 4, 4, 5, COEFFS, 1e-7, 0, None, 0, None) == _lib.ERR_INVALID_ARG
    assert o(p, f32, p, f32, 0, 4, 5, COEFFS, 1e-7, 0, None, 0, None) == _lib.ERR_INVALID_ARG
    assert o(p, f32, p, f32, 4, 4, 5, COEFFS, 1e-7, 0, None, 0, None) == _lib.ERR_WORKSPACE
    assert o(p, bf16, p, bf16, 4, 4, 5, COEFFS, 1e-7, 0, None, 0, None) == _lib.ERR_WORKSPACE
    # element types other than fp32 (0) and bf16 (1) are rejected before anything else is looked at
    for bad_in, bad_out in ((2, f32), (f32, 2), (-1, f32), (f32, 7)):
        assert o(p, bad_in, p, bad_out, 4, 4, 5, COEFFS, 1e-7, 0, None, 0, None) == _lib.ERR_UNSUPPORTED
        assert _lib.lib.muonh_orthogonalize_static(p, bad_in, p, bad_out, 4, 4, 5, COEFFS, 1e-7, 0, None) \
            == _lib.ERR_UNSUPPORTED


def test_workspace_size_layout():
    sz = mh.workspace_size([(256, 128)])
    # X fp32 + 2 X bf16 (128 x 256) + A fp32 + A/B bf16 (128 x 128), plus scalars
    assert sz >= 128 * 256 * (4 + 4) + 128 * 128 * (4 + 4)
    assert sz % 256 == 0
    # a tall and a wide matrix of the same sides share their s x s buffers
    assert mh.workspace_size([(256, 128), (128, 256)]) < 2 * sz + 4096
    # padding: l rounded up to 8 elements
    assert mh.workspace_size([(3, 5)]) >= 3 * 8 * 8
    # grows with the number of matrices, deterministic
    assert mh.workspace_size([(64, 64)] * 10) == mh.workspace_size([(64, 64)] * 10)
    with pytest.raises(mh.MuonHError):
        mh.workspace_size([(0, 3)])


def test_qwen3_2b_workspace_fits():
    import muonh_workloads as wl
    w = wl.qwen3_2b()
    sz = mh.workspace_size(w.shapes)
    assert 10e9 < sz < 20e9
    assert w.n_params == 1_409_286_144


def test_muon_step_rejects_bad_arguments_before_launch():
    good = _arr([(4, 4)])
    m = _lib.lib.muon_step

    def call(arr=good, n=1, lr=0.02, beta=0.95, wd=0.1, steps=5, coeffs=COEFFS, eps=1e-7, flags=0, ws=256,
             ws_bytes=1 << 40):
        return m(arr, n, lr, beta, wd, steps, coeffs, eps, flags, ctypes.c_void_p(ws), ws_bytes, None)

    assert m(None, 1, 0.02, 0.95, 0.1, 5, COEFFS, 1e-7, 0, None, 0, None) == _lib.ERR_INVALID_ARG
    assert call(n=0) == _lib.ERR_INVALID_ARG
    assert call(arr=_arr([(4, 4)], ptr=260)) == _lib.ERR_INVALID_ARG
    assert call(wd=float("inf")) == _lib.ERR_INVALID_ARG
    assert call(lr=float("nan")) == _lib.ERR_INVALID_ARG
    assert call(steps=65) == _lib.ERR_INVALID_ARG
    assert call(flags=0x400) == _lib.ERR_UNSUPPORTED
    assert call(ws=0) == _lib.ERR_WORKSPACE
    assert call(ws_bytes=16) == _lib.ERR_WORKSPACE


def test_adamw_step_rejects_bad_arguments_before_launch():
    def arr(numel=8, ptr=256):
        a = (_lib.AdamParamT * 1)()
        a[0].p = a[0].grad = a[0].exp_avg = a[0].exp_avg_sq = ptr
        a[0].numel = numel
        return a

    f = _lib.lib.adamw_step

    def call(a=None, n=1, step=1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1):
        return f(arr() if a is None else a, n, step, lr, b1, b2, eps, wd, None)

    assert f(None, 1, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1, None) == _lib.ERR_INVALID_ARG
    assert call(n=0) == _lib.ERR_INVALID_ARG
    assert call(step=0) == _lib.ERR_INVALID_ARG
    assert call(b1=1.0) == _lib.ERR_INVALID_ARG
    assert call(b2=-0.1) == _lib.ERR_INVALID_ARG
    assert call(eps=-1.0) == _lib.ERR_INVALID_ARG
    assert call(lr=float("nan")) == _lib.ERR_INVALID_ARG
    assert call(a=arr(numel=0)) == _lib.ERR_INVALID_ARG
    assert call(a=arr(ptr=264)) == _lib.ERR_INVALID_ARG


def test_timeout_hook_rejects_bad_arguments_before_launch():
    ws = ctypes.c_void_p(256)
    f = _lib.lib.muonh_test_gemm_timeout
    assert f(0x1, 1_000_000, ws, _lib.TEST_TIMEOUT_WS_BYTES, None) == _lib.ERR_UNSUPPORTED     # fp32 check
    assert f(0, 10, ws, _lib.TEST_TIMEOUT_WS_BYTES, None) == _lib.ERR_INVALID_ARG             # < 1 us
    assert f(0, 10 ** 11, ws, _lib.TEST_TIMEOUT_WS_BYTES, None) == _lib.ERR_INVALID_ARG       # > 10 s
    assert f(0, 1_000_000, None, _lib.TEST_TIMEOUT_WS_BYTES, None) == _lib.ERR_WORKSPACE
    assert f(0, 1_000_000, ws, _lib.TEST_TIMEOUT_WS_BYTES - 1, None) == _lib.ERR_WORKSPACE
    assert f(0, 1_000_000, ctypes.c_void_p(260), _lib.TEST_TIMEOUT_WS_BYTES, None) == _lib.ERR_WORKSPACE
