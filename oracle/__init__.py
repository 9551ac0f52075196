"""Double-precision CPU oracle for learnable-scale fake-quant (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it; the
two share no code.  The C source (``aqfq_oracle.c``) says which passage of the
pages each step follows.

Arrays are numpy: BF16 tensors travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "aqfq_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "kd_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "libaqfq_oracle.so")
_lock = threading.Lock()
_lib = None

# enums of the oracle (its own copy; the CUDA library defines its own)
INT8, INT4, FP8_E4M3, NVFP4 = 0, 1, 2, 3
PER_TENSOR, PER_CHANNEL, PER_GROUP, PER_HEAD = 0, 1, 2, 3
SCALE_LEARNED, SCALE_DYNAMIC_BLOCK = 0, 1


class Spec(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("fmt", "gran", "group", "qmin", "qmax", "mode")]


def spec(fmt, gran, group=0, qmin=0, qmax=0, mode=SCALE_LEARNED) -> Spec:
    return Spec(fmt, gran, group, qmin, qmax, mode)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available). Returns the .so path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        [os.path.getmtime(f) for f in _SRCS] + [os.path.getmtime(os.path.join(_HERE, "aqfq_oracle.h"))]
    ):
        return _LIB_PATH
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
            "-o", _LIB_PATH + ".tmp", *_SRCS, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_int]
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_decode.argtypes = [ctypes.c_int]
            L.orc_e4m3_encode.restype = ctypes.c_int
            L.orc_e4m3_encode.argtypes = [ctypes.c_double]
            L.orc_e2m1_encode.restype = ctypes.c_int
            L.orc_e2m1_encode.argtypes = [ctypes.c_double]
            L.orc_int_round.restype = ctypes.c_double
            L.orc_int_round.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int]
            L.orc_bf16_round.restype = ctypes.c_uint16
            L.orc_bf16_round.argtypes = [ctypes.c_float]
            L.orc_bf16_value.restype = ctypes.c_float
            L.orc_bf16_value.argtypes = [ctypes.c_uint16]
            L.orc_div32.restype = ctypes.c_float
            L.orc_div32.argtypes = [ctypes.c_float, ctypes.c_float]
            L.orc_qdq_fwd.restype = ctypes.c_int
            L.orc_qdq_fwd.argtypes = [ctypes.POINTER(Spec), P, i64, i64, i64, P, P, P, P, P]
            L.orc_scale_grad.restype = ctypes.c_int
            L.orc_scale_grad.argtypes = [ctypes.POINTER(Spec), P, P, i64, i64, i64, P, P,
                                         P, P, P, P, P]
            L.orc_observer_minmax.restype = ctypes.c_int
            L.orc_observer_minmax.argtypes = [P, i64, i64, i64, P, P, ctypes.c_int]
            L.orc_minmax_scale.restype = ctypes.c_int
            L.orc_minmax_scale.argtypes = [P, P, i64, ctypes.c_double, P]
            L.orc_scale_init.restype = ctypes.c_int
            L.orc_scale_init.argtypes = [ctypes.POINTER(Spec), P, i64, i64, i64, P, P]
            L.orc_num_threads.restype = ctypes.c_int
            L.orc_set_num_threads.restype = None
            L.orc_set_num_threads.argtypes = [ctypes.c_int]
            L.orc_kd_loss.restype = ctypes.c_int
            L.orc_kd_loss.argtypes = [ctypes.c_int, P, P, P, i64, i64, ctypes.c_int32,
                                      ctypes.c_double, ctypes.c_double, P, P, P, P, P, P]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (n >= 1)."""
    lib().orc_set_num_threads(int(n))


# ---- primitives -----------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def int_round(v: float, qmin: int, qmax: int) -> float:
    return lib().orc_int_round(float(v), int(qmin), int(qmax))


def bf16_round(f: float) -> int:
    return int(lib().orc_bf16_round(float(np.float32(f))))


def bf16_value(bits: int) -> float:
    return float(lib().orc_bf16_value(int(bits)))


def div32(a: float, b: float) -> float:
    return float(lib().orc_div32(float(a), float(b)))


# ---- path -----------------------------------------------------------------------

def _shape3(x):
    if x.ndim != 3:
        raise ValueError("expected [batch, rows, K]")
    return x.shape


def qdq_fwd(sp: Spec, x: np.ndarray, scale=None, tensor_scale=None, want_codes=False):
    """x: uint16 [batch, rows, K] BF16 bits. Returns (y bits, codes, block_codes)."""
    x = _c(x, np.uint16)
    B, R, K = _shape3(x)
    y = np.empty_like(x)
    codes = block = None
    if want_codes:
        per_byte = 2 if sp.fmt in (INT4, NVFP4) else 1
        codes = np.zeros((B, R, K // per_byte), np.uint8)
        if sp.fmt == NVFP4:
            block = np.zeros((B, R, K // 16), np.uint8)
    rc = lib().orc_qdq_fwd(ctypes.byref(sp), _p(x), B, R, K, _p(_c(scale, np.float32)),
                           _p(_c(tensor_scale, np.float32)), _p(y), _p(codes), _p(block))
    if rc:
        raise ValueError(f"oracle qdq_fwd rejected the arguments ({rc})")
    return y, codes, block


def scale_grad(sp: Spec, x: np.ndarray, dy: np.ndarray, scale=None, tensor_scale=None):
    """Returns dict: dscale, dscale_abs (float64, scale-shaped), dtensor_scale,
    dtensor_scale_abs (float64 [batch], NVFP4 dynamic only) and dx (uint16 bits)."""
    x = _c(x, np.uint16)
    dy = _c(dy, np.uint16)
    B, R, K = _shape3(x)
    dynamic = sp.fmt == NVFP4 and sp.mode == SCALE_DYNAMIC_BLOCK
    if dynamic:
        nunit = 0
    elif sp.fmt == NVFP4:
        nunit = B * R * (K // 16)
    elif sp.gran == PER_TENSOR:
        nunit = B
    elif sp.gran == PER_CHANNEL:
        nunit = B * R
    elif sp.gran == PER_GROUP:
        nunit = B * R * (K // sp.group)
    else:
        nunit = R
    ds = np.zeros(nunit, np.float64)
    da = np.zeros(nunit, np.float64)
    dt = np.zeros(B, np.float64) if dynamic else None
    dta = np.zeros(B, np.float64) if dynamic else None
    dx = np.empty_like(x)
    rc = lib().orc_scale_grad(ctypes.byref(sp), _p(x), _p(dy), B, R, K,
                              _p(_c(scale, np.float32)), _p(_c(tensor_scale, np.float32)),
                              _p(ds) if nunit else None, _p(da) if nunit else None,
                              _p(dt), _p(dta), _p(dx))
    if rc:
        raise ValueError(f"oracle scale_grad rejected the arguments ({rc})")
    return {"dscale": ds, "dscale_abs": da, "dtensor_scale": dt, "dtensor_scale_abs": dta,
            "dx": dx}


def observer_minmax(x: np.ndarray, mn=None, mx=None):
    """x: uint16 [T, H, D]. If mn/mx are given, merge with them (running min/max)."""
    x = _c(x, np.uint16)
    T, H, D = x.shape
    acc = mn is not None
    lo = np.array(mn, np.float32).copy() if acc else np.empty(H, np.float32)
    hi = np.array(mx, np.float32).copy() if acc else np.empty(H, np.float32)
    rc = lib().orc_observer_minmax(_p(x), T, H, D, _p(lo), _p(hi), int(acc))
    if rc:
        raise ValueError("oracle observer rejected the arguments")
    return lo, hi


def minmax_scale(mn, mx, qmax=448.0):
    mn = _c(mn, np.float32)
    mx = _c(mx, np.float32)
    out = np.empty_like(mn)
    rc = lib().orc_minmax_scale(_p(mn), _p(mx), mn.size, float(qmax), _p(out))
    if rc:
        raise ValueError("oracle minmax_scale rejected the arguments")
    return out


def scale_init(sp: Spec, x: np.ndarray):
    """Returns (scale, tensor_scale) from amax / qmax of each unit."""
    x = _c(x, np.uint16)
    B, R, K = _shape3(x)
    dynamic = sp.fmt == NVFP4 and sp.mode == SCALE_DYNAMIC_BLOCK
    if sp.fmt == NVFP4:
        scale = None if dynamic else np.empty(B * R * (K // 16), np.float32)
        ts = np.empty(B, np.float32)
    else:
        n = {PER_TENSOR: B, PER_CHANNEL: B * R, PER_HEAD: R}.get(sp.gran)
        if n is None:
            n = B * R * (K // sp.group)
        scale = np.empty(n, np.float32)
        ts = None
    rc = lib().orc_scale_init(ctypes.byref(sp), _p(x), B, R, K, _p(scale), _p(ts))
    if rc:
        raise ValueError("oracle scale_init rejected the arguments")
    return scale, ts


def grouped_qdq_gemm(x: np.ndarray, m_offsets, w: np.ndarray, scale, tensor_scale):
    """Reference of the fused NVFP4 fake-quant + grouped GEMM: w_hat from the
    oracle's NVFP4 forward, then y[m] = x[m] . w_hat[e] in double for the rows of
    each expert (a library matmul serves as the contraction step).
    x: uint16 [M, K] BF16 bits; w: uint16 [E, N, K]; returns (y, sum_k |x w_hat|)
    as float64 [M, N]."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    E, N, K = w.shape
    M = x.shape[0]
    sp = spec(NVFP4, PER_GROUP, 16)
    wh, _, _ = qdq_fwd(sp, w, scale, tensor_scale)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (wh.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = np.zeros((M, N), np.float64)
    a = np.zeros((M, N), np.float64)
    off = [int(v) for v in m_offsets]
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            y[lo:hi] = xf[lo:hi] @ wf[e].T
            a[lo:hi] = np.abs(xf[lo:hi]) @ np.abs(wf[e]).T
    return y, a


# ---- distillation losses -----------------------------------------------------------

KD_KL, KD_RKL, KD_CAKLD, KD_MSE = 0, 1, 2, 3


def kd_loss(kd_type, student: np.ndarray, teacher: np.ndarray, labels, topk=0, temperature=1.0,
            grad_scale=1.0, want_grad=True):
    """student, teacher: uint16 [T, V] BF16 bits; labels int [T] (outside [0, V)
    = no loss).  Returns a dict: losses (3,) = means over valid positions of
    (loss, forward KL, backward KL); tok (T, 3) per position; cond (T, 2) error
    scales; dstudent / gmag (T, V) float64 when want_grad; topk_idx (T, K) int32
    when topk > 0."""
    s = _c(student, np.uint16)
    t = _c(teacher, np.uint16)
    lab = _c(labels, np.int32)
    T, V = s.shape
    if t.shape != (T, V) or lab.shape != (T,):
        raise ValueError("shape mismatch")
    losses = np.zeros(3, np.float64)
    tok = np.zeros((T, 3), np.float64)
    cond = np.zeros((T, 2), np.float64)
    ds = np.zeros((T, V), np.float64) if want_grad else None
    gm = np.zeros((T, V), np.float64) if want_grad else None
    idx = np.zeros((T, topk), np.int32) if topk > 0 else None
    rc = lib().orc_kd_loss(int(kd_type), _p(s), _p(t), _p(lab), T, V, int(topk), float(temperature),
                           float(grad_scale), _p(losses), _p(tok), _p(cond), _p(ds), _p(gm), _p(idx))
    if rc:
        raise ValueError(f"oracle kd_loss rejected the arguments ({rc})")
    return {"losses": losses, "tok": tok, "cond": cond, "dstudent": ds, "gmag": gm, "topk_idx": idx}
