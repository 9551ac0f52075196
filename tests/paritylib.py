"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, compare.

Tolerance for scale gradients (stated here, derived in the design notes):
every element term dy * (q - v) is rounded once to binary32 (q - v itself is
exact), then summed in a fixed tree of at most 9 binary32 levels before any
double accumulation, so |gpu - exact| <= 10 * 2^-24 * sum|t| < 1e-6 * sum|t|,
plus the final rounding 2^-24 * |exact|.  A unit passes if
    |gpu - oracle| <= max(1e-5 * |oracle|, 1e-6 * sum|t|),
the 1e-5 relative bar, with the cancellation floor for sums whose terms
cancel (|sum t| << sum|t|).
"""
import numpy as np
import torch

import oracle
from learnable_scale_fake_gb300 import _build, aqfq, synth

REL = 1e-5
FLOOR = 1e-6

_built = False


def dev():
    global _built
    if not _built:
        _build.build()
        aqfq.lib()
        _built = True
    return torch.device("cuda:0")


def ospec(sp):
    return oracle.spec(sp.fmt, sp.gran, sp.group, sp.qmin, sp.qmax, sp.mode)


def bits(t):
    return synth.bf16_bits(t)


def as3(x):
    return x if x.dim() == 3 else x.unsqueeze(0)


def guarded(n, dtype, device, align_elems):
    """A flat buffer with canary bytes on both sides; returns (view, whole)."""
    whole = torch.empty(n + 2 * align_elems, dtype=dtype, device=device)
    whole.view(torch.uint8).fill_(0xA5)
    return whole[align_elems:align_elems + n], whole


def canaries_intact(whole, n, align_elems):
    b = whole.view(torch.uint8)
    esz = whole.element_size()
    head = b[:align_elems * esz]
    tail = b[(align_elems + n) * esz:]
    return bool((head == 0xA5).all()) and bool((tail == 0xA5).all())


def on_device(t, misalign=False):
    """t on the GPU, contiguous; misalign: at an address that is 16-byte but
    not 32-byte aligned (inside a slightly larger buffer)."""
    d = dev()
    if not misalign:
        return t.to(d).contiguous()
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=d)
    v = buf[8:].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


def gpu_fwd(sp, x, scale, ts, codes=True, grouped=False, misalign=False):
    """Runs the forward on the GPU with guard-banded outputs; returns numpy
    (y bits, codes, block codes).  misalign: x and y 16-byte but not 32-byte
    aligned."""
    d = dev()
    x3 = as3(x)
    B, R, K = x3.shape
    xd = on_device(x3, misalign)
    sd = None if scale is None else scale.to(d)
    td = None if ts is None else ts.to(d)
    n = B * R * K
    ya = 72 if misalign else 64  # guard band in elements (144 bytes: 16 mod 32)
    y, yw = guarded(n, torch.bfloat16, d, ya)
    y = y.view(B, R, K)
    c = cw = b = bw = None
    nc = aqfq.codes_numel(sp, B, R, K)
    if codes:
        c, cw = guarded(nc, torch.uint8, d, 256)
        if sp.fmt == aqfq.NVFP4:
            b, bw = guarded(B * R * K // 16, torch.uint8, d, 256)
    if grouped:
        aqfq.aqfq_grouped_qdq(sp, xd, sd, td, y, c, b)
    else:
        aqfq.aqfq_qdq_fwd(sp, xd, sd, td, y, c, b)
    torch.cuda.synchronize()
    assert canaries_intact(yw, n, ya), "write outside y"
    if codes:
        assert canaries_intact(cw, nc, 256), "write outside codes"
        if b is not None:
            assert canaries_intact(bw, B * R * K // 16, 256), "write outside block codes"
    out_c = None if c is None else c.cpu().numpy().reshape(B, R, -1)
    out_b = None if b is None else b.cpu().numpy().reshape(B, R, -1)
    return bits(y), out_c, out_b


def gpu_grad(sp, x, dy, scale, ts, want_dx=True, accumulate_from=None, misalign=False):
    """Runs the scale gradient on the GPU; returns numpy (dscale, dtensor_scale,
    dx bits).  misalign: x, dy and dx 16-byte but not 32-byte aligned."""
    d = dev()
    x3, dy3 = as3(x), as3(dy)
    B, R, K = x3.shape
    xd, dyd = on_device(x3, misalign), on_device(dy3, misalign)
    sd = None if scale is None else scale.to(d)
    td = None if ts is None else ts.to(d)
    dyn = sp.fmt == aqfq.NVFP4 and sp.mode == aqfq.SCALE_DYNAMIC_BLOCK
    n_s = aqfq.scale_numel(sp, B, R, K)
    ds = dts = None
    if dyn:
        dts, dtw = guarded(B, torch.float32, d, 16)
        if accumulate_from is not None:
            dts.copy_(torch.as_tensor(accumulate_from, dtype=torch.float32))
    else:
        ds, dsw = guarded(n_s, torch.float32, d, 16)
        if accumulate_from is not None:
            ds.copy_(torch.as_tensor(accumulate_from, dtype=torch.float32))
    dx = dxw = None
    xa = 72 if misalign else 64
    if want_dx:
        dx, dxw = guarded(B * R * K, torch.bfloat16, d, xa)
        dx = dx.view(B, R, K)
    wsb = aqfq.aqfq_scale_grad_workspace_bytes(sp, B, R, K)
    ws = torch.empty(max(wsb // 8, 1), dtype=torch.float64, device=d) if wsb else None
    aqfq.aqfq_scale_grad(sp, xd, dyd, sd, td, dscale=ds, dtensor_scale=dts, dx=dx,
                         accumulate=accumulate_from is not None, workspace=ws)
    torch.cuda.synchronize()
    if dyn:
        assert canaries_intact(dtw, B, 16)
    else:
        assert canaries_intact(dsw, n_s, 16)
    if want_dx:
        assert canaries_intact(dxw, B * R * K, xa)
    return (None if ds is None else ds.cpu().numpy(), None if dts is None else dts.cpu().numpy(),
            None if dx is None else bits(dx))


def gpu_fwd_grad(sp, x, dy, scale, ts, want_dx=True, misalign=False):
    """The fused forward + gradient on the GPU (guard-banded outputs); returns
    numpy (y bits, dscale, dtensor_scale, dx bits)."""
    d = dev()
    x3, dy3 = as3(x), as3(dy)
    B, R, K = x3.shape
    xd, dyd = on_device(x3, misalign), on_device(dy3, misalign)
    sd = None if scale is None else scale.to(d)
    td = None if ts is None else ts.to(d)
    dyn = sp.fmt == aqfq.NVFP4 and sp.mode == aqfq.SCALE_DYNAMIC_BLOCK
    n = B * R * K
    ga = 72 if misalign else 64
    y, yw = guarded(n, torch.bfloat16, d, ga)
    y = y.view(B, R, K)
    n_s = aqfq.scale_numel(sp, B, R, K)
    ds = dts = None
    if dyn:
        dts, dtw = guarded(B, torch.float32, d, 16)
    else:
        ds, dsw = guarded(n_s, torch.float32, d, 16)
    dx = dxw = None
    if want_dx:
        dx, dxw = guarded(n, torch.bfloat16, d, ga)
        dx = dx.view(B, R, K)
    wsb = aqfq.aqfq_scale_grad_workspace_bytes(sp, B, R, K)
    ws = torch.empty(max(wsb // 8, 1), dtype=torch.float64, device=d) if wsb else None
    aqfq.aqfq_qdq_fwd_grad(sp, xd, dyd, sd, td, y, dscale=ds, dtensor_scale=dts, dx=dx, workspace=ws)
    torch.cuda.synchronize()
    assert canaries_intact(yw, n, ga), "write outside y"
    if dyn:
        assert canaries_intact(dtw, B, 16)
    else:
        assert canaries_intact(dsw, n_s, 16)
    if want_dx:
        assert canaries_intact(dxw, n, ga)
    return (bits(y), None if ds is None else ds.cpu().numpy(), None if dts is None else dts.cpu().numpy(),
            None if dx is None else bits(dx))


def oracle_fwd(sp, x, scale, ts):
    return oracle.qdq_fwd(ospec(sp), bits(as3(x)), None if scale is None else scale.numpy(),
                          None if ts is None else ts.numpy(), True)


def oracle_grad(sp, x, dy, scale, ts):
    return oracle.scale_grad(ospec(sp), bits(as3(x)), bits(as3(dy)),
                             None if scale is None else scale.numpy(),
                             None if ts is None else ts.numpy())


def assert_grad_close(got, ref, ref_abs, extra_abs=None, what="dscale"):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    floor = FLOOR * (ref_abs if extra_abs is None else ref_abs + np.abs(extra_abs))
    tol = np.maximum(REL * np.abs(ref), floor)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, (f"{what}: {bad.size}/{err.size} units beyond tolerance; worst "
                           f"rel {np.max(err / np.maximum(np.abs(ref), 1e-300)):.3g}, e.g. unit "
                           f"{bad[0]}: gpu {got[bad[0]]!r} oracle {ref[bad[0]]!r} "
                           f"sum|t| {ref_abs[bad[0]]!r}")
    return float(np.mean(err <= REL * np.abs(ref))) if err.size else 1.0
