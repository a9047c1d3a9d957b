"""MuonH optimizer step (momentum -> Newton-Schulz -> hyperball projection)
on B300 (sm_103a), behind the C ABI in include/muonh.h.

MuonH, as the Puro-2B digest (jacksunwei.me) describes it in "The load-bearing
tricks aren't in the abstract": Muon's orthogonalised-momentum update, with
every weight matrix held at the Frobenius norm it had at initialisation.

PyTorch supplies device memory and the current stream; every step of the
computation runs in libmuonh's CUDA kernels.

    opt = MuonH(weights, lr=0.02)        # fp32 2-D CUDA tensors; captures r0
    ...backward...
    opt.step()                           # uses w.grad, or opt.step(grads)
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (FLAG_FP32_CHECK, FLAG_GEMM_1SM, FLAG_GEMM_ONE_STEP, FLAG_ONE_STREAM, FLAG_GRAD_BF16, FLAG_NESTEROV, FLAG_SCALE_RMS,  # noqa: F401
                   FLAG_SCALE_SHAPE,
                   FLAG_SYNC_DEBUG, STATUS_DEGENERATE_NORM, STATUS_KERNEL_TIMEOUT, STATUS_NONFINITE_INPUT,
                   MuonHError, check, lib)

NS_COEFFS = (3.4445, -4.7750, 2.0315)

__all__ = ["MuonH", "Muon", "AdamW", "ShardedMuonH", "partition", "exchange_weights", "adamw_step", "capture_norms", "workspace_size", "step", "muon_step", "orthogonalize",
           "orthogonalize_workspace_size", "get_status", "profile_read", "MuonHError", "NS_COEFFS"]


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check_tensor(t, name, dtype=torch.float32):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def matrix_array(weights, grads=None, moms=None, bf16=None, grad_dtype=torch.float32):
    """Build the muonh_matrix_t array for a list of 2-D tensors (gradients
    bfloat16 when the step runs with MUONH_FLAG_GRAD_BF16)."""
    n = len(weights)
    arr = (_lib.MatrixT * n)()
    for i, w in enumerate(weights):
        if w.dim() != 2:
            raise ValueError(f"matrix {i} is not 2-D")
        _check_tensor(w, f"weights[{i}]")
        arr[i].w = w.data_ptr()
        arr[i].rows, arr[i].cols = w.shape
        if grads is not None:
            _check_tensor(grads[i], f"grads[{i}]", grad_dtype)
            arr[i].grad = grads[i].data_ptr()
        if moms is not None:
            _check_tensor(moms[i], f"moms[{i}]")
            arr[i].mom = moms[i].data_ptr()
        if bf16 is not None and bf16[i] is not None:
            _check_tensor(bf16[i], f"bf16[{i}]", torch.bfloat16)
            arr[i].w_bf16 = bf16[i].data_ptr()
    return arr


def capture_norms(weights, out=None, stream=None) -> torch.Tensor:
    """r0[i] = ||weights[i]||_F (fp32 CUDA tensor), via muonh_capture_norms."""
    arr = matrix_array(weights)
    if out is None:
        out = torch.empty(len(weights), dtype=torch.float32, device=weights[0].device)
    check(lib.muonh_capture_norms(arr, len(weights), ctypes.c_void_p(out.data_ptr()), _stream(stream)),
          "muonh_capture_norms")
    return out


def workspace_size(shapes_or_arr, flags: int = 0) -> int:
    if isinstance(shapes_or_arr, ctypes.Array):
        arr = shapes_or_arr
    else:
        arr = (_lib.MatrixT * len(shapes_or_arr))()
        for i, (r, c) in enumerate(shapes_or_arr):
            arr[i].rows, arr[i].cols = r, c
            arr[i].w = 256  # any aligned non-null value: only shapes are read
    out = ctypes.c_size_t()
    check(lib.muonh_workspace_size(arr, len(arr), flags, ctypes.byref(out)), "muonh_workspace_size")
    return out.value


def step(arr, r0, lr, beta, ns_steps, coeffs, eps, flags, workspace, stream=None) -> None:
    """One muonh_step call on a prebuilt matrix array."""
    c = (ctypes.c_float * 3)(*coeffs)
    check(lib.muonh_step(arr, len(arr), ctypes.c_void_p(r0.data_ptr()), lr, beta, ns_steps, c, eps, flags,
                         ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream(stream)),
          "muonh_step")


def muon_step(arr, lr, beta, weight_decay, ns_steps, coeffs, eps, flags, workspace, stream=None) -> None:
    """One muon_step call (plain Muon, decoupled weight decay) on a prebuilt matrix array."""
    c = (ctypes.c_float * 3)(*coeffs)
    check(lib.muon_step(arr, len(arr), lr, beta, weight_decay, ns_steps, c, eps, flags,
                        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream(stream)), "muon_step")


def orthogonalize_workspace_size(rows: int, cols: int, flags: int = 0) -> int:
    out = ctypes.c_size_t()
    check(lib.muonh_orthogonalize_workspace_size(rows, cols, flags, ctypes.byref(out)),
          "muonh_orthogonalize_workspace_size")
    return out.value


def _dtype_code(t, name):
    if not t.is_cuda or not t.is_contiguous() or t.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"{name} must be a contiguous CUDA float32 or bfloat16 tensor")
    return _lib.DTYPE_F32 if t.dtype == torch.float32 else _lib.DTYPE_BF16


def orthogonalize(x: torch.Tensor, ns_steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7,
                  flags: int = 0, out=None, workspace=None, stream=None, out_dtype=torch.float32) -> torch.Tensor:
    """Newton-Schulz of a fp32 or bf16 CUDA matrix (muonh_orthogonalize);
    the result is fp32 unless ``out_dtype`` (or ``out``) says bf16."""
    in_code = _dtype_code(x, "x")
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    out_code = _dtype_code(out, "out")
    r, c_ = x.shape
    need = orthogonalize_workspace_size(r, c_, flags)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    cf = (ctypes.c_float * 3)(*coeffs)
    check(lib.muonh_orthogonalize(ctypes.c_void_p(x.data_ptr()), in_code, ctypes.c_void_p(out.data_ptr()), out_code,
                                  r, c_, ns_steps, cf, eps, flags, ctypes.c_void_p(workspace.data_ptr()),
                                  workspace.numel(), _stream(stream)), "muonh_orthogonalize")
    return out


def orthogonalize_static(x: torch.Tensor, ns_steps: int = 5, coeffs=NS_COEFFS, eps: float = 1e-7,
                         flags: int = 0, out=None, stream=None, out_dtype=torch.float32) -> torch.Tensor:
    """Newton-Schulz without a workspace (muonh_orthogonalize_static).

    For code that cannot allocate device memory: scratch comes from the
    library's fixed device array (see include/muonh.h).  ``out`` must be
    given by such callers; calls that may overlap on the GPU race.
    """
    in_code = _dtype_code(x, "x")
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    out_code = _dtype_code(out, "out")
    r, c_ = x.shape
    cf = (ctypes.c_float * 3)(*coeffs)
    check(lib.muonh_orthogonalize_static(ctypes.c_void_p(x.data_ptr()), in_code, ctypes.c_void_p(out.data_ptr()),
                                         out_code, r, c_, ns_steps, cf, eps, flags, _stream(stream)),
          "muonh_orthogonalize_static")
    return out


def get_status(stream=None) -> int:
    """Synchronise, read and clear the device status word."""
    v = ctypes.c_uint32()
    check(lib.muonh_get_status(ctypes.byref(v), _stream(stream)), "muonh_get_status")
    return v.value


def profile_read() -> dict:
    """Per-kernel totals recorded since muonh_profile_enable(1) (blocking)."""
    buf = (_lib.ProfileEntry * 32)()
    n = ctypes.c_int()
    check(lib.muonh_profile_read(buf, 32, ctypes.byref(n)), "muonh_profile_read")
    return {buf[i].name.decode(): {"launches": buf[i].launches, "ms": buf[i].ms, "flops": buf[i].flops,
                                   "bytes": buf[i].bytes} for i in range(n.value)}


class MuonH:
    """MuonH over a fixed list of fp32 2-D CUDA weight matrices.

    r0 (the radius each matrix is held at) is captured from the weights at
    construction; momenta start at zero.  ``bf16_copies=True`` keeps a bf16
    copy of every weight, refreshed by each step.
    """

    def __init__(self, weights, lr=0.02, beta=0.95, ns_steps=5, ns_coeffs=NS_COEFFS, eps=1e-7,
                 bf16_copies=False, fp32_check=False, flags=0):
        self.weights = list(weights)
        self.lr, self.beta, self.ns_steps, self.eps = float(lr), float(beta), int(ns_steps), float(eps)
        self.ns_coeffs = tuple(float(v) for v in ns_coeffs)
        self.flags = (FLAG_FP32_CHECK if fp32_check else 0) | int(flags)
        self.moms = [torch.zeros_like(w) for w in self.weights]
        self.bf16 = [torch.empty_like(w, dtype=torch.bfloat16) for w in self.weights] if bf16_copies else None
        self.r0 = capture_norms(self.weights)
        self._arrays = {}
        self.workspace = torch.empty(workspace_size([tuple(w.shape) for w in self.weights], self.flags),
                                     dtype=torch.uint8, device=self.weights[0].device)

    def step(self, grads=None, stream=None) -> None:
        if grads is None:
            grads = [w.grad for w in self.weights]
        step(self._array_for(grads), self.r0, self.lr, self.beta, self.ns_steps, self.ns_coeffs, self.eps,
             self.flags, self.workspace, stream)

    def _array_for(self, grads):
        # one matrix array per set of gradient buffers (a few at most): a
        # training loop that alternates buffers rebuilds nothing
        ptrs = tuple(g.data_ptr() for g in grads)
        arr = self._arrays.get(ptrs)
        if arr is None:
            if len(self._arrays) >= 4:
                self._arrays.clear()
            arr = self._arrays[ptrs] = matrix_array(
                self.weights, grads, self.moms, self.bf16,
                torch.bfloat16 if self.flags & FLAG_GRAD_BF16 else torch.float32)
        return arr

    def state_dict(self):
        return {"moms": [m.clone() for m in self.moms], "r0": self.r0.clone()}

    def load_state_dict(self, sd):
        for m, src in zip(self.moms, sd["moms"]):
            m.copy_(src)
        self.r0.copy_(sd["r0"])


class Muon:
    """Plain Muon (the baseline MuonH is compared with) over a fixed list of
    fp32 2-D CUDA weight matrices: momentum, Newton-Schulz, then
    W <- (1 - lr*weight_decay)*W - lr*O.  Momenta start at zero."""

    def __init__(self, weights, lr=0.02, beta=0.95, weight_decay=0.0, ns_steps=5, ns_coeffs=NS_COEFFS, eps=1e-7,
                 bf16_copies=False, fp32_check=False, flags=0):
        self.weights = list(weights)
        self.lr, self.beta, self.weight_decay = float(lr), float(beta), float(weight_decay)
        self.ns_steps, self.eps = int(ns_steps), float(eps)
        self.ns_coeffs = tuple(float(v) for v in ns_coeffs)
        self.flags = (FLAG_FP32_CHECK if fp32_check else 0) | int(flags)
        self.moms = [torch.zeros_like(w) for w in self.weights]
        self.bf16 = [torch.empty_like(w, dtype=torch.bfloat16) for w in self.weights] if bf16_copies else None
        self._arrays = {}
        self.workspace = torch.empty(workspace_size([tuple(w.shape) for w in self.weights], self.flags),
                                     dtype=torch.uint8, device=self.weights[0].device)

    def step(self, grads=None, stream=None) -> None:
        if grads is None:
            grads = [w.grad for w in self.weights]
        muon_step(self._array_for(grads), self.lr, self.beta, self.weight_decay, self.ns_steps, self.ns_coeffs,
                  self.eps, self.flags, self.workspace, stream)

    def _array_for(self, grads):
        ptrs = tuple(g.data_ptr() for g in grads)
        arr = self._arrays.get(ptrs)
        if arr is None:
            if len(self._arrays) >= 4:
                self._arrays.clear()
            arr = self._arrays[ptrs] = matrix_array(
                self.weights, grads, self.moms, self.bf16,
                torch.bfloat16 if self.flags & FLAG_GRAD_BF16 else torch.float32)
        return arr


def adamw_array(params, grads, exp_avgs, exp_avg_sqs, bf16=None):
    """Build the adamw_param_t array for lists of contiguous fp32 CUDA tensors."""
    arr = (_lib.AdamParamT * len(params))()
    for i, p in enumerate(params):
        for t, nm in ((p, "params"), (grads[i], "grads"), (exp_avgs[i], "exp_avgs"), (exp_avg_sqs[i], "exp_avg_sqs")):
            if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError(f"{nm}[{i}] must be a contiguous CUDA float32 tensor")
        arr[i].p, arr[i].grad = p.data_ptr(), grads[i].data_ptr()
        arr[i].exp_avg, arr[i].exp_avg_sq = exp_avgs[i].data_ptr(), exp_avg_sqs[i].data_ptr()
        arr[i].numel = p.numel()
        if bf16 is not None and bf16[i] is not None:
            arr[i].p_bf16 = bf16[i].data_ptr()
    return arr


def adamw_step(arr, step, lr, beta1, beta2, eps, weight_decay, stream=None) -> None:
    """One adamw_step call on a prebuilt adamw_param_t array."""
    check(lib.adamw_step(arr, len(arr), int(step), lr, beta1, beta2, eps, weight_decay, _stream(stream)),
          "adamw_step")


class AdamW:
    """AdamW (decoupled weight decay, bias-corrected moments) over a fixed
    list of contiguous fp32 CUDA tensors: the optimizer of the parameters
    outside the MuonH group.  Moments start at zero."""

    def __init__(self, params, lr=2e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, bf16_copies=False):
        self.params = list(params)
        self.lr, self.eps, self.weight_decay = float(lr), float(eps), float(weight_decay)
        self.beta1, self.beta2 = (float(b) for b in betas)
        self.exp_avgs = [torch.zeros_like(p) for p in self.params]
        self.exp_avg_sqs = [torch.zeros_like(p) for p in self.params]
        self.bf16 = [torch.empty_like(p, dtype=torch.bfloat16) for p in self.params] if bf16_copies else None
        self.t = 0
        self._arrays = {}

    def step(self, grads=None, stream=None) -> None:
        if grads is None:
            grads = [p.grad for p in self.params]
        ptrs = tuple(g.data_ptr() for g in grads)
        arr = self._arrays.get(ptrs)
        if arr is None:
            if len(self._arrays) >= 4:
                self._arrays.clear()
            arr = self._arrays[ptrs] = adamw_array(self.params, grads, self.exp_avgs, self.exp_avg_sqs, self.bf16)
        self.t += 1
        adamw_step(arr, self.t, self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, stream)


from .sharded import ShardedMuonH, exchange_weights, partition  # noqa: E402
