"""ctypes binding of libmuonh.so: argument marshalling only.

Every computation runs in the library's CUDA kernels; this module turns
torch tensors into device pointers, the current torch stream into a
cudaStream_t and return codes into exceptions.  There is no other code path:
if the shared library is missing, importing this module fails.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmuonh.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_WORKSPACE = 2
ERR_UNSUPPORTED = 3
ERR_CUDA = 4

STATUS_NONFINITE_INPUT = 0x1
STATUS_DEGENERATE_NORM = 0x2
STATUS_KERNEL_TIMEOUT = 0x4

FLAG_FP32_CHECK = 0x1
FLAG_NESTEROV = 0x2
FLAG_SYNC_DEBUG = 0x4
FLAG_GEMM_1SM = 0x8
FLAG_GEMM_ONE_STEP = 0x100
FLAG_ONE_STREAM = 0x200
FLAG_SCALE_SHAPE = 0x10
FLAG_SCALE_RMS = 0x20
FLAG_GRAD_BF16 = 0x40

MAX_SIDE = 65536

DTYPE_F32 = 0
DTYPE_BF16 = 1

# Every symbol include/muonh.h declares.
EXPORTS = (
    "muonh_capture_norms", "muonh_workspace_size", "muonh_step",
    "muonh_orthogonalize_workspace_size", "muonh_orthogonalize", "muonh_get_status",
    "muonh_status_string", "muonh_last_error", "muonh_version",
    "muonh_profile_enable", "muonh_profile_read", "muonh_launch_count",
    "muonh_orthogonalize_static", "muon_step", "adamw_step", "muonh_partition",
    "muonh_test_gemm_timeout",
)

STATIC_SCRATCH_BYTES = 96 * 1024 * 1024
TEST_TIMEOUT_WS_BYTES = 512 * 1024


class MatrixT(ctypes.Structure):
    """muonh_matrix_t"""
    _fields_ = [
        ("w", ctypes.c_void_p),
        ("w_bf16", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("mom", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
    ]


class AdamParamT(ctypes.Structure):
    """adamw_param_t"""
    _fields_ = [
        ("p", ctypes.c_void_p),
        ("p_bf16", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("exp_avg", ctypes.c_void_p),
        ("exp_avg_sq", ctypes.c_void_p),
        ("numel", ctypes.c_int64),
    ]


class ProfileEntry(ctypes.Structure):
    """muonh_profile_entry_t"""
    _fields_ = [
        ("name", ctypes.c_char_p),
        ("launches", ctypes.c_int64),
        ("ms", ctypes.c_double),
        ("flops", ctypes.c_double),
        ("bytes", ctypes.c_double),
    ]


class MuonHError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        super().__init__(f"{where}: {detail} (code {code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python hyperball_constrained_muon_muonh_b300/build.py` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, U32, SZ, F, I64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t,
                             ctypes.c_float, ctypes.c_int64)
    mp = ctypes.POINTER(MatrixT)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.muonh_capture_norms.argtypes = [mp, I, P, P]
    lib.muonh_workspace_size.argtypes = [mp, I, U32, ctypes.POINTER(SZ)]
    lib.muonh_step.argtypes = [mp, I, P, F, F, I, fp, F, U32, P, SZ, P]
    lib.muon_step.argtypes = [mp, I, F, F, F, I, fp, F, U32, P, SZ, P]
    lib.adamw_step.argtypes = [ctypes.POINTER(AdamParamT), I, I, F, F, F, F, F, P]
    lib.muonh_partition.argtypes = [mp, I, I, ctypes.POINTER(I)]
    lib.muonh_orthogonalize_workspace_size.argtypes = [I64, I64, U32, ctypes.POINTER(SZ)]
    lib.muonh_orthogonalize.argtypes = [P, I, P, I, I64, I64, I, fp, F, U32, P, SZ, P]
    lib.muonh_orthogonalize_static.argtypes = [P, I, P, I, I64, I64, I, fp, F, U32, P]
    lib.muonh_get_status.argtypes = [ctypes.POINTER(U32), P]
    lib.muonh_status_string.argtypes = [I]
    lib.muonh_status_string.restype = ctypes.c_char_p
    lib.muonh_last_error.argtypes = []
    lib.muonh_last_error.restype = ctypes.c_char_p
    lib.muonh_version.argtypes = []
    lib.muonh_profile_enable.argtypes = [I]
    lib.muonh_profile_read.argtypes = [ctypes.POINTER(ProfileEntry), I, ctypes.POINTER(I)]
    lib.muonh_launch_count.argtypes = []
    lib.muonh_test_gemm_timeout.argtypes = [U32, ctypes.c_uint64, P, SZ, P]
    for name in EXPORTS:
        if name not in ("muonh_status_string", "muonh_last_error"):
            getattr(lib, name).restype = ctypes.c_int
    lib.muonh_launch_count.restype = ctypes.c_int64
    return lib


lib = _load()


def check(code: int, where: str) -> None:
    if code != OK:
        detail = lib.muonh_last_error().decode() or lib.muonh_status_string(code).decode()
        raise MuonHError(code, where, detail)
