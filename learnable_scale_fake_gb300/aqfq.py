"""Thin ctypes binding of libaqfq (include/aqfq.h): argument marshalling only.

Every function has the name of the C entry point it calls and takes torch
tensors already on the GPU (PyTorch only provides device memory and
streams); outputs are caller-allocated tensors that the call fills.  The
CUDA library must be built (``__graft_entry__.build()`` or
``python -m learnable_scale_fake_gb300._build``); there is no fallback: if it
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libaqfq.so")

# enums of include/aqfq.h
INT8, INT4, FP8_E4M3, NVFP4 = 0, 1, 2, 3
PER_TENSOR, PER_CHANNEL, PER_GROUP, PER_HEAD = 0, 1, 2, 3
SCALE_LEARNED, SCALE_DYNAMIC_BLOCK = 0, 1
KD_KL, KD_RKL, KD_CAKLD, KD_MSE = 0, 1, 2, 3

STATUS = {0: "AQFQ_OK", 1: "AQFQ_ERR_NULL", 2: "AQFQ_ERR_SHAPE", 3: "AQFQ_ERR_ALIGN",
          4: "AQFQ_ERR_UNSUPPORTED", 5: "AQFQ_ERR_WORKSPACE", 6: "AQFQ_ERR_CUDA"}

# every symbol include/aqfq.h declares
EXPORTS = ("aqfq_qdq_fwd", "aqfq_grouped_qdq", "aqfq_grouped_qdq_gemm", "aqfq_scale_grad",
           "aqfq_qdq_fwd_grad", "aqfq_scale_grad_noalloc",
           "aqfq_scale_grad_workspace_bytes", "aqfq_observer_minmax", "aqfq_minmax_scale",
           "aqfq_scale_init", "aqfq_kd_loss", "aqfq_kd_workspace_bytes",
           "aqfq_selftest_wait_timeout", "aqfq_selftest_grid_codes", "aqfq_status_string",
           "aqfq_version")


class QSpec(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("fmt", "gran", "group", "qmin", "qmax", "mode")]


def qspec(fmt, gran, group=0, qmin=0, qmax=0, mode=SCALE_LEARNED) -> QSpec:
    return QSpec(fmt, gran, group, qmin, qmax, mode)


class AqfqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


_lock = threading.Lock()
_lib = None


def lib():
    """Load libaqfq.so (raises if it is missing: no CPU fallback exists)."""
    global _lib
    if _lib is not None:  # loaded: no lock needed to read the reference
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libaqfq.so is not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            S = ctypes.POINTER(QSpec)
            sig = {
                "aqfq_qdq_fwd": (i32, [S, P, i64, i64, i64, P, P, P, P, P, P]),
                "aqfq_grouped_qdq": (i32, [S, P, i64, i64, i64, P, P, P, P, P, P]),
                "aqfq_grouped_qdq_gemm": (i32, [P, P, i64, P, P, P, i64, i64, i64, P, P, P]),
                "aqfq_scale_grad": (i32, [S, P, P, i64, i64, i64, P, P, P, P, P, i32, P, sz, P]),
                "aqfq_qdq_fwd_grad": (i32, [S, P, P, i64, i64, i64, P, P, P, P, P, P, i32, P, sz,
                                            P]),
                "aqfq_scale_grad_noalloc": (i32, [S, P, P, i64, i64, i64, P, P, P, P, P, i32, P]),
                "aqfq_scale_grad_workspace_bytes": (sz, [S, i64, i64, i64]),
                "aqfq_observer_minmax": (i32, [P, i64, i64, i64, P, P, i32, P]),
                "aqfq_minmax_scale": (i32, [P, P, i64, ctypes.c_float, P, P]),
                "aqfq_scale_init": (i32, [S, P, i64, i64, i64, P, P, P]),
                "aqfq_kd_loss": (i32, [i32, P, P, P, i64, i64, ctypes.c_int32, ctypes.c_float,
                                       ctypes.c_float, P, P, P, P, P, sz, P]),
                "aqfq_kd_workspace_bytes": (sz, [i64]),
                "aqfq_selftest_wait_timeout": (i32, [P, ctypes.c_uint32, P]),
                "aqfq_selftest_grid_codes": (i32, [S, P, i64, P, P]),
                "aqfq_status_string": (ctypes.c_char_p, [i32]),
                "aqfq_version": (i32, []),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("aqfq works on CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("aqfq needs contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, status):
    if status != 0:
        raise AqfqError(fn, status)


def _bf16(t, name):
    if t is not None and t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")


def _f32(t, name):
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")


def _u8(t, name):
    if t is not None and t.dtype != torch.uint8:
        raise TypeError(f"{name} must be uint8")


def _brk(x):
    """[batch, rows, K] of a 2D or 3D tensor."""
    if x.dim() == 2:
        return 1, x.shape[0], x.shape[1]
    if x.dim() == 3:
        return x.shape
    raise ValueError("expected a [rows, K] or [batch, rows, K] tensor")


def aqfq_qdq_fwd(spec, x, scale, tensor_scale, y, codes=None, block_codes=None, stream=None):
    _bf16(x, "x"), _bf16(y, "y"), _f32(scale, "scale"), _f32(tensor_scale, "tensor_scale")
    _u8(codes, "codes"), _u8(block_codes, "block_codes")
    B, R, K = _brk(x)
    st = lib().aqfq_qdq_fwd(ctypes.byref(spec), _ptr(x), B, R, K, _ptr(scale), _ptr(tensor_scale),
                            _ptr(y), _ptr(codes), _ptr(block_codes), _stream(stream))
    _check("aqfq_qdq_fwd", st)


def aqfq_grouped_qdq(spec, w, scale, tensor_scale, y, codes=None, block_codes=None, stream=None):
    _bf16(w, "w"), _bf16(y, "y"), _f32(scale, "scale"), _f32(tensor_scale, "tensor_scale")
    _u8(codes, "codes"), _u8(block_codes, "block_codes")
    if w.dim() != 3:
        raise ValueError("w must be an [E, N, K] stack")
    E, N, K = w.shape
    st = lib().aqfq_grouped_qdq(ctypes.byref(spec), _ptr(w), E, N, K, _ptr(scale),
                                _ptr(tensor_scale), _ptr(y), _ptr(codes), _ptr(block_codes),
                                _stream(stream))
    _check("aqfq_grouped_qdq", st)


def aqfq_grouped_qdq_gemm(x, m_offsets, w, scale, tensor_scale, y, error_flag=None, stream=None):
    """y[m] = x[m] @ w_hat[e].T for the rows m of expert e (m_offsets int32 [E+1])."""
    _bf16(x, "x"), _bf16(w, "w"), _bf16(y, "y"), _f32(scale, "scale")
    _f32(tensor_scale, "tensor_scale")
    if m_offsets.dtype != torch.int32 or (error_flag is not None and error_flag.dtype != torch.int32):
        raise TypeError("m_offsets and error_flag must be int32")
    if w.dim() != 3 or x.dim() != 2:
        raise ValueError("x must be [total_m, K] and w [E, N, K]")
    E, N, K = w.shape
    st = lib().aqfq_grouped_qdq_gemm(_ptr(x), _ptr(m_offsets), x.shape[0], _ptr(w), _ptr(scale),
                                     _ptr(tensor_scale), E, N, K, _ptr(y), _ptr(error_flag),
                                     _stream(stream))
    _check("aqfq_grouped_qdq_gemm", st)


def aqfq_selftest_wait_timeout(flag, polls, stream=None):
    """Diagnostic: a bounded device wait that nothing completes sets flag (int32
    device tensor) to 1 after `polls` polls."""
    if flag.dtype != torch.int32:
        raise TypeError("flag must be int32")
    _check("aqfq_selftest_wait_timeout",
           lib().aqfq_selftest_wait_timeout(_ptr(flag), int(polls), _stream(stream)))


def aqfq_selftest_grid_codes(spec, v, codes, stream=None):
    """Diagnostic: the kernels' grid-rounding code of every binary32 value of v
    (float32 device tensor) into codes (uint8, same length)."""
    _f32(v, "v"), _u8(codes, "codes")
    if codes.numel() != v.numel():
        raise ValueError("codes must have one byte per value")
    _check("aqfq_selftest_grid_codes",
           lib().aqfq_selftest_grid_codes(ctypes.byref(spec), _ptr(v), v.numel(), _ptr(codes),
                                          _stream(stream)))


def aqfq_kd_workspace_bytes(T) -> int:
    return int(lib().aqfq_kd_workspace_bytes(int(T)))


def aqfq_kd_loss(kd_type, student, teacher, labels, losses, workspace, topk=0, temperature=1.0,
                 grad_scale=1.0, token_loss=None, dstudent=None, topk_idx=None, stream=None):
    """Distillation loss of student against teacher logits [T, V] (BF16) with
    labels int32 [T]; fills losses float32 [3] (loss, forward KL, backward KL),
    and optionally token_loss [T], dstudent [T, V] BF16 and topk_idx int32 [T, topk].
    workspace: a uint8 device tensor of aqfq_kd_workspace_bytes(T) bytes."""
    _bf16(student, "student"), _bf16(teacher, "teacher"), _bf16(dstudent, "dstudent")
    _f32(losses, "losses"), _f32(token_loss, "token_loss"), _u8(workspace, "workspace")
    if labels.dtype != torch.int32 or (topk_idx is not None and topk_idx.dtype != torch.int32):
        raise TypeError("labels and topk_idx must be int32")
    if student.dim() != 2 or teacher.shape != student.shape:
        raise ValueError("student and teacher must both be [T, V]")
    T, V = student.shape
    st = lib().aqfq_kd_loss(int(kd_type), _ptr(student), _ptr(teacher), _ptr(labels), T, V,
                            int(topk), float(temperature), float(grad_scale), _ptr(losses),
                            _ptr(token_loss), _ptr(dstudent), _ptr(topk_idx), _ptr(workspace),
                            workspace.numel(), _stream(stream))
    _check("aqfq_kd_loss", st)


def aqfq_scale_grad_workspace_bytes(spec, batch, rows, K) -> int:
    return int(lib().aqfq_scale_grad_workspace_bytes(ctypes.byref(spec), batch, rows, K))


def aqfq_scale_grad(spec, x, dy, scale, tensor_scale, dscale=None, dtensor_scale=None, dx=None,
                    accumulate=False, workspace=None, stream=None):
    _bf16(x, "x"), _bf16(dy, "dy"), _bf16(dx, "dx")
    _f32(scale, "scale"), _f32(tensor_scale, "tensor_scale")
    _f32(dscale, "dscale"), _f32(dtensor_scale, "dtensor_scale")
    B, R, K = _brk(x)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().aqfq_scale_grad(ctypes.byref(spec), _ptr(x), _ptr(dy), B, R, K, _ptr(scale),
                               _ptr(tensor_scale), _ptr(dscale), _ptr(dtensor_scale), _ptr(dx),
                               int(bool(accumulate)), _ptr(workspace), wsb, _stream(stream))
    _check("aqfq_scale_grad", st)


def aqfq_qdq_fwd_grad(spec, x, dy, scale, tensor_scale, y, dscale=None, dtensor_scale=None,
                      dx=None, accumulate=False, workspace=None, stream=None):
    """Forward (y = x_hat) and scale gradient of the same tensor in one pass."""
    _bf16(x, "x"), _bf16(dy, "dy"), _bf16(dx, "dx"), _bf16(y, "y")
    _f32(scale, "scale"), _f32(tensor_scale, "tensor_scale")
    _f32(dscale, "dscale"), _f32(dtensor_scale, "dtensor_scale")
    B, R, K = _brk(x)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().aqfq_qdq_fwd_grad(ctypes.byref(spec), _ptr(x), _ptr(dy), B, R, K, _ptr(scale),
                                 _ptr(tensor_scale), _ptr(y), _ptr(dscale), _ptr(dtensor_scale),
                                 _ptr(dx), int(bool(accumulate)), _ptr(workspace), wsb,
                                 _stream(stream))
    _check("aqfq_qdq_fwd_grad", st)


def aqfq_scale_grad_noalloc(spec, x, dy, scale, tensor_scale, dscale=None, dtensor_scale=None,
                            dx=None, accumulate=False, stream=None):
    """aqfq_scale_grad without a workspace argument, for callers that cannot
    allocate device memory: the library's built-in 128 KiB scratch is used."""
    _bf16(x, "x"), _bf16(dy, "dy"), _bf16(dx, "dx")
    _f32(scale, "scale"), _f32(tensor_scale, "tensor_scale")
    _f32(dscale, "dscale"), _f32(dtensor_scale, "dtensor_scale")
    B, R, K = _brk(x)
    st = lib().aqfq_scale_grad_noalloc(ctypes.byref(spec), _ptr(x), _ptr(dy), B, R, K, _ptr(scale),
                                       _ptr(tensor_scale), _ptr(dscale), _ptr(dtensor_scale),
                                       _ptr(dx), int(bool(accumulate)), _stream(stream))
    _check("aqfq_scale_grad_noalloc", st)


def aqfq_observer_minmax(x, min_out, max_out, accumulate=False, stream=None):
    _bf16(x, "x"), _f32(min_out, "min_out"), _f32(max_out, "max_out")
    if x.dim() != 3:
        raise ValueError("x must be [T, H, D]")
    T, H, D = x.shape
    st = lib().aqfq_observer_minmax(_ptr(x), T, H, D, _ptr(min_out), _ptr(max_out),
                                    int(bool(accumulate)), _stream(stream))
    _check("aqfq_observer_minmax", st)


def aqfq_minmax_scale(min_in, max_in, qmax, scale_out, stream=None):
    _f32(min_in, "min_in"), _f32(max_in, "max_in"), _f32(scale_out, "scale_out")
    st = lib().aqfq_minmax_scale(_ptr(min_in), _ptr(max_in), min_in.numel(), float(qmax),
                                 _ptr(scale_out), _stream(stream))
    _check("aqfq_minmax_scale", st)


def aqfq_scale_init(spec, x, scale, tensor_scale, stream=None):
    _bf16(x, "x"), _f32(scale, "scale"), _f32(tensor_scale, "tensor_scale")
    B, R, K = _brk(x)
    st = lib().aqfq_scale_init(ctypes.byref(spec), _ptr(x), B, R, K, _ptr(scale),
                               _ptr(tensor_scale), _stream(stream))
    _check("aqfq_scale_init", st)


def aqfq_status_string(status: int) -> str:
    return lib().aqfq_status_string(int(status)).decode()


def aqfq_version() -> int:
    return int(lib().aqfq_version())


# ---- shape helpers (no arithmetic of the method) -------------------------------------

def scale_numel(spec, batch, rows, K) -> int:
    """Number of learned scales the spec uses for an x of [batch, rows, K]."""
    if spec.fmt == NVFP4:
        return 0 if spec.mode == SCALE_DYNAMIC_BLOCK else batch * rows * (K // 16)
    return {PER_TENSOR: batch, PER_CHANNEL: batch * rows, PER_HEAD: rows}.get(
        spec.gran, batch * rows * (K // max(spec.group, 1)))


def codes_numel(spec, batch, rows, K) -> int:
    return batch * rows * (K // 2 if spec.fmt in (INT4, NVFP4) else K)

