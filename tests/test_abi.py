"""The C ABI on the host: the library loads, exports every entry point that
include/aqfq.h declares, and rejects bad arguments before any launch (the
checks run before any kernel, so fake pointer values are safe here).  One
test (marked gpu) checks the workspace sizes, which follow the current
device's SM count."""
import ctypes
import os
import re

import pytest
import torch

from learnable_scale_fake_gb300 import _build, aqfq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, NULL, SHAPE, ALIGN, UNSUP, WS, CUDA = 0, 1, 2, 3, 4, 5, 6
A = 0x10000  # a fake, 256-byte aligned "device" address


@pytest.fixture(scope="module")
def L():
    _build.build()
    return aqfq.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "aqfq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(aqfq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(aqfq.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {aqfq.LIB_PATH}").read()
    for name in header_functions():
        assert re.search(rf"\bT {name}\b", out), name


def test_status_strings_and_version(L):
    assert aqfq.aqfq_version() == 100
    for s in range(7):
        assert aqfq.aqfq_status_string(s)
    assert aqfq.aqfq_status_string(99) == "unknown status"


def fwd(L, spec, x=A, B=1, R=4, K=64, scale=A, ts=A, y=2 * A, codes=None, blk=None):
    sp = None if spec is None else ctypes.byref(spec)
    return L.aqfq_qdq_fwd(sp, x, B, R, K, scale, ts, y, codes, blk, None)


def grad(L, spec, x=A, dy=2 * A, B=1, R=4, K=64, scale=A, ts=A, ds=3 * A, dts=None, dx=None,
         ws=None, wsb=0):
    return L.aqfq_scale_grad(ctypes.byref(spec), x, dy, B, R, K, scale, ts, ds, dts, dx, 0, ws,
                             wsb, None)


NV = aqfq.qspec(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
NVD = aqfq.qspec(aqfq.NVFP4, aqfq.PER_GROUP, group=16, mode=aqfq.SCALE_DYNAMIC_BLOCK)
I8 = aqfq.qspec(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127)
I4 = aqfq.qspec(aqfq.INT4, aqfq.PER_GROUP, group=128, qmin=-8, qmax=7)
F8T = aqfq.qspec(aqfq.FP8_E4M3, aqfq.PER_TENSOR)


def test_forward_argument_checks(L):
    assert fwd(L, None) == NULL
    assert fwd(L, NV, x=None) == NULL
    assert fwd(L, NV, y=None) == NULL
    assert fwd(L, NV, ts=None) == NULL
    assert fwd(L, NV, scale=None) == NULL
    assert fwd(L, NV, K=24) == SHAPE
    assert fwd(L, NV, R=-1) == SHAPE
    assert fwd(L, NV, x=A + 8) == ALIGN           # BF16 tensors: 16-byte aligned at least
    assert fwd(L, I8, y=A + 24) == ALIGN
    assert fwd(L, NV, y=A + 2) == ALIGN
    assert fwd(L, NV, scale=A + 2) == ALIGN
    assert fwd(L, NV, codes=A + 4, blk=A) == ALIGN
    assert fwd(L, NV, codes=A) == NULL          # NVFP4 codes come with block codes
    assert fwd(L, I8, codes=A + 8) == ALIGN      # byte codes are 16-byte aligned
    assert fwd(L, I8, blk=A, codes=A) == UNSUP   # block codes are NVFP4 only
    assert fwd(L, I4, K=192) == SHAPE            # K % group
    assert fwd(L, I8, K=20) == SHAPE             # K % 8
    assert fwd(L, I4, K=136) == SHAPE            # K = 8 * odd: no group or block formats
    assert fwd(L, I8, K=24, codes=A + 4) == ALIGN  # 8-element chunks: byte codes 8-byte aligned
    I4C = aqfq.qspec(aqfq.INT4, aqfq.PER_CHANNEL, qmin=-8, qmax=7)
    assert fwd(L, I4C, K=24, codes=A + 2) == ALIGN  # and nibble codes 4-byte aligned
    assert fwd(L, aqfq.qspec(aqfq.NVFP4, aqfq.PER_GROUP, group=32)) == UNSUP
    assert fwd(L, aqfq.qspec(aqfq.NVFP4, aqfq.PER_CHANNEL, group=16)) == UNSUP
    assert fwd(L, aqfq.qspec(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-129, qmax=127)) == UNSUP
    assert fwd(L, aqfq.qspec(aqfq.INT4, aqfq.PER_CHANNEL, qmin=-8, qmax=8)) == UNSUP
    assert fwd(L, aqfq.qspec(aqfq.INT4, aqfq.PER_GROUP, group=96, qmin=-8, qmax=7), K=192) == UNSUP
    assert fwd(L, aqfq.qspec(aqfq.FP8_E4M3, aqfq.PER_GROUP, group=1024), K=1024) == UNSUP
    assert fwd(L, aqfq.qspec(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127, mode=1)) == UNSUP
    assert fwd(L, aqfq.qspec(7, aqfq.PER_CHANNEL)) == UNSUP
    assert fwd(L, NV, R=1 << 30, K=1 << 10) == SHAPE  # rows * K / 16 >= 2^32
    assert fwd(L, NVD, scale=None, x=A + 8) == ALIGN  # dynamic mode needs no block scales


def test_grouped_and_init_argument_checks(L):
    assert L.aqfq_grouped_qdq(ctypes.byref(NV), A, 2, 4, 48, A, None, 2 * A, None, None, None) == NULL
    assert L.aqfq_grouped_qdq(ctypes.byref(NV), A, 2, 4, 40, A, A, 2 * A, None, None, None) == SHAPE
    assert L.aqfq_scale_init(ctypes.byref(I8), None, 1, 4, 64, A, None, None) == NULL
    assert L.aqfq_scale_init(ctypes.byref(I8), A + 1, 1, 4, 64, A, None, None) == ALIGN
    assert L.aqfq_scale_init(ctypes.byref(NV), A, 1, 4, 64, A, None, None) == NULL


def test_grad_argument_checks(L):
    assert grad(L, NV, ds=None) == NULL
    assert grad(L, NV, dts=A) == UNSUP            # learned NVFP4 has a fixed tensor scale
    assert grad(L, NVD, scale=None) == NULL       # needs dtensor_scale
    assert grad(L, NVD, scale=None, ds=A, dts=A) == UNSUP
    assert grad(L, NV, dy=A + 8) == ALIGN
    assert grad(L, NV, dx=A + 8) == ALIGN
    assert aqfq.aqfq_scale_grad_workspace_bytes(NV, 1, 4, 40) == 0  # rejected shape


def fused(L, spec, x=A, dy=2 * A, B=1, R=4, K=64, scale=A, ts=A, y=4 * A, ds=3 * A, dts=None,
          dx=None, ws=None, wsb=0):
    return L.aqfq_qdq_fwd_grad(ctypes.byref(spec), x, dy, B, R, K, scale, ts, y, ds, dts, dx, 0, ws,
                               wsb, None)


def test_fused_argument_checks(L):
    """aqfq_qdq_fwd_grad checks what aqfq_scale_grad checks, plus y."""
    assert L.aqfq_qdq_fwd_grad(None, A, A, 1, 4, 64, A, A, A, A, None, None, 0, None, 0, None) == NULL
    assert fused(L, NV, y=None) == NULL
    assert fused(L, NV, y=4 * A + 8) == ALIGN
    assert fused(L, NV, ds=None) == NULL
    assert fused(L, NV, dts=A) == UNSUP
    assert fused(L, NV, K=24) == SHAPE
    assert fused(L, NV, dy=A + 8) == ALIGN
    assert fused(L, I8, K=20) == SHAPE
    # an empty tensor needs no buffers
    assert fused(L, NV, B=0, x=None, dy=None, y=None, ds=None, ts=None) in (OK, CUDA)


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers pass the checks: no device only")
def test_boundary_accepts_rows_of_eight_and_sixteen_byte_alignment(L):
    """K % 8 == 0 rows (per-tensor / per-channel / per-head INT8, INT4, FP8) and
    BF16 tensors that are 16-byte but not 32-byte aligned pass every host
    check; without a device the call then fails at the launch (AQFQ_ERR_CUDA)."""
    I4C = aqfq.qspec(aqfq.INT4, aqfq.PER_CHANNEL, qmin=-8, qmax=7)
    F8H = aqfq.qspec(aqfq.FP8_E4M3, aqfq.PER_HEAD)
    CUDA_ = 6
    assert fwd(L, I8, K=24) == CUDA_
    assert fwd(L, I8, K=8, codes=A + 8) == CUDA_
    assert fwd(L, I4C, K=56, codes=A + 4) == CUDA_
    assert fwd(L, F8T, K=40) == CUDA_
    assert fwd(L, F8H, K=24) == CUDA_
    assert fwd(L, NV, x=A + 16, y=A + 48) == CUDA_
    assert fwd(L, I4, K=128, x=A + 16) == CUDA_
    assert grad(L, I8, K=24, dx=A + 16) == CUDA_
    assert grad(L, NV, x=A + 16, dy=A + 48) == CUDA_
    assert L.aqfq_observer_minmax(A + 16, 4, 2, 24, A, 2 * A, 0, None) == CUDA_
    assert L.aqfq_scale_init(ctypes.byref(I8), A + 16, 1, 4, 24, A, None, None) == CUDA_
    assert fused(L, I8, K=24, y=4 * A + 16) == CUDA_
    assert fused(L, NVD, scale=None, ds=None, dts=A, ws=5 * A, wsb=1 << 20) == CUDA_


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a device")
def test_grad_without_a_device_is_a_cuda_error(L):
    """Grids and workspaces follow the device's SM count: with no device to
    query, the workspace bound is 0 and a call with valid arguments returns
    AQFQ_ERR_CUDA instead of guessing a size (nothing is launched)."""
    assert aqfq.aqfq_scale_grad_workspace_bytes(NVD, 1, 4, 64) == 0
    assert aqfq.aqfq_scale_grad_workspace_bytes(F8T, 3, 4, 64) == 0
    assert grad(L, NVD, scale=None, ds=None, dts=A) == CUDA
    assert grad(L, NV) == CUDA


@pytest.mark.gpu
def test_grad_workspace_checks(L):
    """Workspace sizes and their checks (they follow the current device's SM
    count); every call here is rejected on the host before any launch."""
    torch.zeros(1, device="cuda")  # a current device
    assert grad(L, NVD, scale=None, ds=None, dts=A) == WS
    need = aqfq.aqfq_scale_grad_workspace_bytes(NVD, 1, 4, 64)
    assert need > 0 and need % 8 == 0
    assert grad(L, NVD, scale=None, ds=None, dts=A, ws=A, wsb=need - 8) == WS
    assert grad(L, NVD, scale=None, ds=None, dts=A, ws=A + 4, wsb=need) == ALIGN
    hd = aqfq.qspec(aqfq.FP8_E4M3, aqfq.PER_HEAD)
    assert grad(L, hd) == WS                      # per-head sums need a workspace
    assert aqfq.aqfq_scale_grad_workspace_bytes(hd, 1000, 4, 64) == 1000 * 16 * 8  # all tokens
    big = aqfq.aqfq_scale_grad_workspace_bytes(hd, 100000, 4, 64)  # one wave of the device
    assert big % (16 * 8) == 0 and 16 * 8 <= big < 100000 * 16 * 8
    assert aqfq.aqfq_scale_grad_workspace_bytes(I8, 1, 4, 64) == 0
    assert aqfq.aqfq_scale_grad_workspace_bytes(I4, 2, 8, 128) == 0
    assert aqfq.aqfq_scale_grad_workspace_bytes(F8T, 3, 4, 64) == 16 + 3 * 8  # counter + partials


def test_observer_argument_checks(L):
    f = L.aqfq_observer_minmax
    assert f(A, 4, 2, 12, A, 2 * A, 0, None) == SHAPE
    assert f(A, -1, 2, 16, A, 2 * A, 0, None) == SHAPE
    assert f(None, 4, 2, 16, A, 2 * A, 0, None) == NULL
    assert f(A + 8, 4, 2, 16, A, 2 * A, 0, None) == ALIGN
    assert f(A, 4, 2, 20, A, 2 * A, 0, None) == SHAPE   # D % 8
    assert f(A, 4, 1 << 21, 256, A, 2 * A, 0, None) == SHAPE
    m = L.aqfq_minmax_scale
    assert m(A, A, 4, ctypes.c_float(0.0), A, None) == SHAPE
    assert m(A, None, 4, ctypes.c_float(448.0), A, None) == NULL
    assert m(A, A + 2, 4, ctypes.c_float(448.0), A, None) == ALIGN


def test_grid_codes_diagnostic_checks(L):
    f = L.aqfq_selftest_grid_codes
    assert f(None, A, 4, A, None) == NULL
    assert f(ctypes.byref(I8), None, 4, A, None) == NULL
    assert f(ctypes.byref(I8), A, -1, A, None) == SHAPE
    assert f(ctypes.byref(I8), A + 2, 4, A, None) == ALIGN
    assert f(ctypes.byref(aqfq.qspec(7, 0)), A, 4, A, None) == UNSUP
    assert f(ctypes.byref(aqfq.qspec(aqfq.INT4, 0, qmin=-9, qmax=7)), A, 4, A, None) == UNSUP
    assert f(ctypes.byref(I8), None, 0, None, None) == OK  # nothing to do


def test_fastdiv_constants_exhaustive_small():
    """The host constants of the multiply-shift division (Granlund-Montgomery
    round-up method) reproduce n // d; checked here in Python for the divisors
    the kernels use (K / 16 up to 2^20) over edge numerators."""
    def consts(d):
        l = (d - 1).bit_length()
        m = ((1 << 32) * ((1 << l) - d)) // d + 1
        return m, min(l, 1), max(l - 1, 0)

    def div(n, d):
        m, s1, s2 = consts(d)
        t = (m * n) >> 32
        return (t + ((n - t) >> s1)) >> s2

    import random
    rnd = random.Random(0)
    ds = list(range(1, 600)) + [rnd.randrange(1, 1 << 20) for _ in range(300)] + [(1 << 20)]
    for d in ds:
        for n in [0, 1, d - 1, d, d + 1, 2 * d - 1, (1 << 32) - 1, (1 << 32) - d] + \
                 [rnd.randrange(0, 1 << 32) for _ in range(20)]:
            if 0 <= n < (1 << 32):
                assert div(n, d) == n // d, (n, d)


def kd(L, kd_type=0, s=A, t=2 * A, lab=3 * A, T=4, V=64, topk=0, tau=1.0, gs=1.0, losses=4 * A,
       tl=None, ds=None, idx=None, ws=5 * A, wsb=1 << 20):
    return L.aqfq_kd_loss(kd_type, s, t, lab, T, V, topk, tau, gs, losses, tl, ds, idx, ws, wsb, None)


def test_kd_loss_host_checks(L):
    assert kd(L, kd_type=4) == UNSUP
    assert kd(L, kd_type=-1) == UNSUP
    assert kd(L, V=60) == SHAPE            # V % 8
    assert kd(L, V=0) == SHAPE
    assert kd(L, T=-1) == SHAPE
    assert kd(L, topk=65) == SHAPE         # topk > V
    assert kd(L, topk=-1) == SHAPE
    assert kd(L, tau=0.0) == SHAPE
    assert kd(L, tau=-2.0) == SHAPE
    assert kd(L, tau=float("inf")) == SHAPE
    assert kd(L, gs=float("nan")) == SHAPE
    assert kd(L, kd_type=3, topk=5) == UNSUP       # mse: no top-K
    assert kd(L, kd_type=3, tau=2.0) == UNSUP      # mse: no temperature
    assert kd(L, idx=6 * A) == UNSUP               # topk_idx needs topk > 0
    assert kd(L, losses=None) == NULL
    assert kd(L, s=None) == NULL
    assert kd(L, lab=None) == NULL
    assert kd(L, ws=None) == WS
    assert kd(L, wsb=aqfq.aqfq_kd_workspace_bytes(4) - 1) == WS
    assert kd(L, s=A + 8) == ALIGN
    assert kd(L, ds=6 * A + 4) == ALIGN
    assert kd(L, tl=6 * A + 2) == ALIGN
    assert aqfq.aqfq_kd_workspace_bytes(0) == 1024
    assert aqfq.aqfq_kd_workspace_bytes(4096) >= 1024 + 12 * 4096


def test_selftest_wait_timeout_host_checks(L):
    assert L.aqfq_selftest_wait_timeout(None, 16, None) == NULL
    assert L.aqfq_selftest_wait_timeout(A + 2, 16, None) == ALIGN
    assert L.aqfq_selftest_wait_timeout(A, 0, None) == SHAPE
    assert L.aqfq_selftest_wait_timeout(A, (1 << 22) + 1, None) == SHAPE
