"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element
by element, on seeded inputs that span several CTA tiles with ragged tails.
Codes, dequantised values, block codes and min/max must match bit for bit;
scale gradients within the tolerance stated in paritylib."""
import numpy as np
import pytest
import torch

import oracle
from learnable_scale_fake_gb300 import aqfq, synth
from paritylib import (as3, assert_grad_close, bits, dev, gpu_fwd, gpu_fwd_grad, gpu_grad,
                       oracle_fwd, oracle_grad, ospec)

pytestmark = pytest.mark.gpu

Q = aqfq.qspec
NV = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
NVD = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16, mode=aqfq.SCALE_DYNAMIC_BLOCK)


def _x_normal(shape, seed):
    return synth.normal_bf16(shape, 0.02, seed)


def _x_t(shape, seed):
    return synth.student_t_outliers_bf16(shape, 4, 0.02, 5e-3, 20.0, seed)


def _x_act(shape, seed):
    return synth.normal_outliers_bf16(shape, 1.0, 1e-2, 30.0, seed)


# name, spec, (B, R, K), x generator, scale range, tensor-scale range
CASES = [
    ("int8_channel_k512", Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), (2, 33, 512),
     _x_normal, (1e-4, 4e-4), None),
    ("int8_channel_k128", Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), (3, 45, 128),
     _x_normal, (1e-4, 4e-4), None),
    ("int8_channel_k528", Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), (2, 19, 528),
     _x_normal, (1e-4, 4e-4), None),
    ("int8_sym_tensor", Q(aqfq.INT8, aqfq.PER_TENSOR, qmin=-127, qmax=127), (3, 21, 256),
     _x_normal, (1e-4, 4e-4), None),
    ("int4_g128", Q(aqfq.INT4, aqfq.PER_GROUP, group=128, qmin=-8, qmax=7), (2, 29, 384),
     _x_normal, (2e-3, 2e-2), None),
    ("int4_g16", Q(aqfq.INT4, aqfq.PER_GROUP, group=16, qmin=-8, qmax=7), (2, 21, 240),
     _x_normal, (2e-3, 2e-2), None),
    ("int4_g512_sym", Q(aqfq.INT4, aqfq.PER_GROUP, group=512, qmin=-7, qmax=7), (2, 9, 1024),
     _x_normal, (2e-3, 2e-2), None),
    ("fp8_channel", Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL), (2, 37, 272), _x_normal, (2e-5, 2e-4),
     None),
    ("fp8_tensor", Q(aqfq.FP8_E4M3, aqfq.PER_TENSOR), (3, 23, 352), _x_normal, (2e-5, 2e-4),
     None),
    ("fp8_g32", Q(aqfq.FP8_E4M3, aqfq.PER_GROUP, group=32), (2, 27, 320), _x_normal,
     (2e-5, 2e-4), None),
    ("fp8_head", Q(aqfq.FP8_E4M3, aqfq.PER_HEAD), (97, 6, 64), _x_normal, (2e-5, 2e-4), None),
    ("int8_sym_head", Q(aqfq.INT8, aqfq.PER_HEAD, qmin=-127, qmax=127), (61, 5, 48), _x_normal,
     (1e-4, 4e-4), None),
    ("nvfp4_learned", NV, (3, 45, 208), _x_t, (2e-3, 2e-2), (2e-5, 1e-4)),
    ("nvfp4_dynamic", NVD, (3, 41, 192), _x_act, None, (1e-4, 1e-2)),
    # rows of K = 8 * odd elements (8-element chunks, 128-bit accesses)
    ("int8_channel_k24", Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), (2, 37, 24),
     _x_normal, (1e-4, 4e-4), None),
    ("int8_channel_k8", Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), (2, 41, 8),
     _x_normal, (1e-4, 4e-4), None),
    ("fp8_channel_k520", Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL), (1, 23, 520), _x_normal,
     (2e-5, 2e-4), None),
    ("int4_channel_k56", Q(aqfq.INT4, aqfq.PER_CHANNEL, qmin=-8, qmax=7), (2, 19, 56),
     _x_normal, (2e-3, 2e-2), None),
    ("int8_tensor_k40", Q(aqfq.INT8, aqfq.PER_TENSOR, qmin=-128, qmax=127), (3, 17, 40),
     _x_normal, (1e-4, 4e-4), None),
    ("fp8_head_d24", Q(aqfq.FP8_E4M3, aqfq.PER_HEAD), (53, 5, 24), _x_normal, (2e-5, 2e-4), None),
    # long rows: one CTA per row for the per-channel gradient (513 chunks of 8: a ragged tail)
    ("fp8_channel_k4104", Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL), (1, 7, 4104), _x_normal,
     (2e-5, 2e-4), None),
    ("int8_channel_k4096", Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), (2, 5, 4096),
     _x_normal, (1e-4, 4e-4), None),
]
IDS = [c[0] for c in CASES]


def _inputs(case, seed=0):
    name, sp, shape, xg, srange, trange = case
    B, R, K = shape
    x = xg(shape, seed + 1)
    dy = synth.normal_bf16(shape, 1.0, seed + 2)
    n = aqfq.scale_numel(sp, B, R, K)
    scale = synth.loguniform_f32((n,), *srange, seed + 3) if srange else None
    ts = synth.loguniform_f32((B,), *trange, seed + 4) if trange else None
    return x, dy, scale, ts


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_forward_bit_exact(case):
    sp = case[1]
    x, _, scale, ts = _inputs(case)
    y, c, b = gpu_fwd(sp, x, scale, ts)
    y_ref, c_ref, b_ref = oracle_fwd(sp, x, scale, ts)
    assert np.array_equal(y, y_ref), f"{np.count_nonzero(y != y_ref)} x_hat mismatches"
    assert np.array_equal(c, c_ref), f"{np.count_nonzero(c != c_ref)} code mismatches"
    if sp.fmt == aqfq.NVFP4:
        assert np.array_equal(b, b_ref)
    # the forward without code outputs writes the same values
    y2, _, _ = gpu_fwd(sp, x, scale, ts, codes=False)
    assert np.array_equal(y2, y_ref)


@pytest.mark.parametrize("case", [c for c in CASES if c[1].fmt == aqfq.NVFP4],
                         ids=[c[0] for c in CASES if c[1].fmt == aqfq.NVFP4])
def test_grouped_entry_equals_forward(case):
    sp = case[1]
    x, _, scale, ts = _inputs(case, seed=10)
    y, c, b = gpu_fwd(sp, x, scale, ts, grouped=True)
    y_ref, c_ref, b_ref = oracle_fwd(sp, x, scale, ts)
    assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref) and np.array_equal(b, b_ref)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_scale_grad(case):
    sp = case[1]
    x, dy, scale, ts = _inputs(case)
    ds, dts, dx = gpu_grad(sp, x, dy, scale, ts)
    ref = oracle_grad(sp, x, dy, scale, ts)
    if sp.fmt == aqfq.NVFP4 and sp.mode == aqfq.SCALE_DYNAMIC_BLOCK:
        assert_grad_close(dts, ref["dtensor_scale"], ref["dtensor_scale_abs"], what="dtensor_scale")
    else:
        frac = assert_grad_close(ds, ref["dscale"], ref["dscale_abs"])
        print(f"{case[0]}: {frac:.4f} of units within plain 1e-5 relative")
    assert np.array_equal(dx, ref["dx"]), f"{np.count_nonzero(dx != ref['dx'])} dx mismatches"


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fused_forward_and_gradient(case):
    """aqfq_qdq_fwd_grad: one pass writes the forward's x_hat (bit-exact) and
    the scale gradient (within the tolerance) and dx (bit-exact), as the two
    separate entry points do; 16-byte aligned views for every third case."""
    sp = case[1]
    x, dy, scale, ts = _inputs(case, seed=5)
    mis = IDS.index(case[0]) % 3 == 0
    y, ds, dts, dx = gpu_fwd_grad(sp, x, dy, scale, ts, misalign=mis)
    y_ref, _, _ = oracle_fwd(sp, x, scale, ts)
    ref = oracle_grad(sp, x, dy, scale, ts)
    assert np.array_equal(y, y_ref), f"{np.count_nonzero(y != y_ref)} x_hat mismatches"
    if dts is not None:
        assert_grad_close(dts, ref["dtensor_scale"], ref["dtensor_scale_abs"], what="dtensor_scale")
    else:
        assert_grad_close(ds, ref["dscale"], ref["dscale_abs"])
    assert np.array_equal(dx, ref["dx"])
    # without the STE input gradient: the same x_hat and scale gradient
    y2, ds2, dts2, _ = gpu_fwd_grad(sp, x, dy, scale, ts, want_dx=False)
    assert np.array_equal(y2, y_ref)
    got, want = (ds2, ds) if ds is not None else (dts2, dts)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), "not reproducible"


ACC = [c for c in CASES if c[0] in ("int8_channel_k512", "int4_g128", "fp8_tensor", "fp8_head",
                                    "nvfp4_learned", "nvfp4_dynamic", "fp8_channel_k4104")]


@pytest.mark.parametrize("case", ACC, ids=[c[0] for c in ACC])
def test_scale_grad_accumulate_and_determinism(case):
    sp = case[1]
    x, dy, scale, ts = _inputs(case, seed=20)
    ds1, dts1, _ = gpu_grad(sp, x, dy, scale, ts, want_dx=False)
    ds2, dts2, _ = gpu_grad(sp, x, dy, scale, ts, want_dx=False)
    first = ds1 if ds1 is not None else dts1
    second = ds2 if ds2 is not None else dts2
    assert np.array_equal(first.view(np.uint32), second.view(np.uint32)), "not reproducible"
    ref = oracle_grad(sp, x, dy, scale, ts)
    dyn = sp.fmt == aqfq.NVFP4 and sp.mode == aqfq.SCALE_DYNAMIC_BLOCK
    r, ra = (ref["dtensor_scale"], ref["dtensor_scale_abs"]) if dyn else (ref["dscale"], ref["dscale_abs"])
    old = synth.loguniform_f32(r.shape, 1e-3, 10.0, seed=21).numpy() * np.where(
        np.arange(r.size) % 2, 1, -1).astype(np.float32)
    ds, dts, _ = gpu_grad(sp, x, dy, scale, ts, want_dx=False, accumulate_from=old)
    got = ds if ds is not None else dts
    assert_grad_close(got, old.astype(np.float64) + r, ra, extra_abs=old, what="accumulated")


SIXTEEN = [c for c in CASES if c[0] in ("int8_channel_k512", "int8_channel_k528", "int4_g128",
                                         "fp8_tensor", "fp8_head", "nvfp4_learned", "nvfp4_dynamic",
                                         "int8_channel_k24", "fp8_head_d24")]


@pytest.mark.parametrize("case", SIXTEEN, ids=[c[0] for c in SIXTEEN])
def test_sixteen_byte_aligned_views(case):
    """x, y, dy and dx at addresses that are 16-byte but not 32-byte aligned
    (a row slice of a wider tensor, for instance): the 128-bit access path
    gives the same codes, values and gradients as the oracle."""
    sp = case[1]
    x, dy, scale, ts = _inputs(case, seed=25)
    y, c, b = gpu_fwd(sp, x, scale, ts, misalign=True)
    y_ref, c_ref, b_ref = oracle_fwd(sp, x, scale, ts)
    assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref)
    if sp.fmt == aqfq.NVFP4:
        assert np.array_equal(b, b_ref)
    ds, dts, dx = gpu_grad(sp, x, dy, scale, ts, misalign=True)
    ref = oracle_grad(sp, x, dy, scale, ts)
    if dts is not None:
        assert_grad_close(dts, ref["dtensor_scale"], ref["dtensor_scale_abs"], what="dtensor_scale")
    else:
        assert_grad_close(ds, ref["dscale"], ref["dscale_abs"])
    assert np.array_equal(dx, ref["dx"])


@pytest.mark.parametrize("name", ["fp8_tensor", "nvfp4_dynamic"])
def test_reduced_grad_batch_beyond_grid_limit(name):
    """Per-tensor and NVFP4 tensor-scale gradients over 70000 batch entries
    (above the 65535 grid-y limit: a CTA walks several entries, and the last
    CTA to finish adds every entry's partials)."""
    case = next(c for c in CASES if c[0] == name)
    case = (case[0], case[1], (70000, 1, 32)) + case[3:]
    sp = case[1]
    x, dy, scale, ts = _inputs(case, seed=30)
    ds, dts, _ = gpu_grad(sp, x, dy, scale, ts, want_dx=False)
    ref = oracle_grad(sp, x, dy, scale, ts)
    if dts is not None:
        assert_grad_close(dts, ref["dtensor_scale"], ref["dtensor_scale_abs"], what="dtensor_scale")
    else:
        assert_grad_close(ds, ref["dscale"], ref["dscale_abs"])


def test_per_head_grad_many_rounds():
    """x [T, H, D] large enough that each thread of the per-head gradient walks
    several tokens (more chunks than threads), with the STE input gradient."""
    sp = Q(aqfq.FP8_E4M3, aqfq.PER_HEAD)
    T, H, D = 20000, 8, 128
    x = synth.head_normal_bf16(T, H, D, 0.1, 10.0, seed=95)
    dy = synth.normal_bf16((T, H, D), 1.0, seed=96)
    s = synth.loguniform_f32((H,), 2e-4, 2e-2, seed=97)
    ds, _, dx = gpu_grad(sp, x, dy, s, None)
    ref = oracle_grad(sp, x, dy, s, None)
    assert_grad_close(ds, ref["dscale"], ref["dscale_abs"])
    assert np.array_equal(dx, ref["dx"])


def test_special_values():
    """Zero scales, all-zero blocks, signed zeros, saturation, BF16 subnormals,
    exact halfway points: every format, forward and gradient."""
    B, R, K = 2, 8, 256
    g = torch.Generator().manual_seed(3)
    x = synth.normal_bf16((B, R, K), 0.02, seed=30)
    xf = x.float()
    xf[0, 0, :16] = 0.0
    xf[0, 1, :16] = -0.0
    xf[0, 2, 0:8] = torch.tensor([1e-39, -1e-39, 3e-40, -5e-41, 1e-38, 9e-39, -2e-39, 0.0])
    xf[1, 3, :] = 1e4
    xf[1, 4, :] = -3e38
    x = xf.to(torch.bfloat16)
    dy = synth.normal_bf16((B, R, K), 1.0, seed=31)
    specs = [(Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), (1e-4, 4e-4)),
             (Q(aqfq.INT4, aqfq.PER_GROUP, group=128, qmin=-8, qmax=7), (2e-3, 2e-2)),
             (Q(aqfq.FP8_E4M3, aqfq.PER_GROUP, group=16), (2e-5, 2e-4)),
             (NV, (2e-3, 2e-2))]
    for sp, rng in specs:
        n = aqfq.scale_numel(sp, B, R, K)
        s = synth.loguniform_f32((n,), *rng, seed=32)
        s[::5] = 0.0                                   # zero scales
        s[1::7] = 2.0 ** torch.randint(-12, -4, ((n - 1 + 6) // 7,), generator=g).float()
        ts = torch.tensor([3e-5, 0.0], dtype=torch.float32) if sp.fmt == aqfq.NVFP4 else None
        y, c, b = gpu_fwd(sp, x, s, ts)
        y_ref, c_ref, b_ref = oracle_fwd(sp, x, s, ts)
        assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref)
        if b is not None:
            assert np.array_equal(b, b_ref)
        ds, _, dx = gpu_grad(sp, x, dy, s, ts)
        ref = oracle_grad(sp, x, dy, s, ts)
        assert_grad_close(ds, ref["dscale"], ref["dscale_abs"])
        assert np.array_equal(dx, ref["dx"])
        # the fused pass gives the same x_hat and gradients on these values too
        yf, dsf, _, dxf = gpu_fwd_grad(sp, x, dy, s, ts)
        assert np.array_equal(yf, y_ref) and np.array_equal(dxf, ref["dx"])
        assert_grad_close(dsf, ref["dscale"], ref["dscale_abs"])
    # scales at and beyond the ends of the reciprocal fast path [2^-64, 2^64],
    # with BF16 subnormal and tiny inputs: forward bit-exact, gradient in tolerance
    edge = torch.tensor([2.0 ** -64, 2.0 ** -64 * (1 - 2 ** -24), 2.0 ** 64, 2.0 ** 64 * (1 + 2 ** -23),
                         3.1e-20, 7.7e18, 1e-30, 1e30], dtype=torch.float32)
    xe = synth.normal_bf16((1, 8, 64), 1.0, seed=33).float()
    xe[:, :, :16] *= 1e-36                        # tiny and subnormal BF16 values
    xe[:, :, 16:32] *= 1e-20
    xe[:, :, 32:48] *= 1e20
    xe = xe.to(torch.bfloat16)
    dye = synth.normal_bf16((1, 8, 64), 1.0, seed=34)
    for sp in (Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL)):
        y, c, _ = gpu_fwd(sp, xe, edge, None)
        y_ref, c_ref, _ = oracle_fwd(sp, xe, edge, None)
        assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref)
        ds, _, dx = gpu_grad(sp, xe, dye, edge, None)
        ref = oracle_grad(sp, xe, dye, edge, None)
        assert_grad_close(ds, ref["dscale"], ref["dscale_abs"])
        assert np.array_equal(dx, ref["dx"])
        yf, dsf, _, dxf = gpu_fwd_grad(sp, xe, dye, edge, None)
        assert np.array_equal(yf, y_ref) and np.array_equal(dxf, ref["dx"])
        assert_grad_close(dsf, ref["dscale"], ref["dscale_abs"])
    sb = edge.repeat_interleave(4)                 # NVFP4: block scale = S_b / g * g
    for g in (1.0, 2.0 ** -30):
        ts = torch.tensor([g], dtype=torch.float32)
        y, c, b = gpu_fwd(NV, xe, sb * g, ts)
        y_ref, c_ref, b_ref = oracle_fwd(NV, xe, sb * g, ts)
        assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref) and np.array_equal(b, b_ref)
    # exact ties of the integer grid: x = (k + 1/2) * s with s a power of two
    s = torch.full((R,), 2.0 ** -8)
    k = torch.arange(-140, 140, dtype=torch.float32)
    xt = ((k[: K] + 0.5) * 2.0 ** -8).repeat(R, 1)[:, :K].to(torch.bfloat16).unsqueeze(0)
    sp = Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127)
    y, c, _ = gpu_fwd(sp, xt, s, None)
    y_ref, c_ref, _ = oracle_fwd(sp, xt, s, None)
    assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref)


def test_all_bf16_values_through_each_grid():
    """Every finite BF16 pattern through E4M3 (scale 1) and E2M1 (block scale 1),
    and through INT8 with scale 1: the hardware conversions against the
    oracle's grid enumeration; then the same values under random scales."""
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (allb.astype(np.uint32) << 16).view(np.float32)
    allb = allb[np.isfinite(f)]
    allb = allb[: allb.size // 16 * 16]
    x = synth.from_bits(allb.reshape(1, -1, 16))
    one = torch.ones(1, dtype=torch.float32)
    for sp, s, ts in [(Q(aqfq.FP8_E4M3, aqfq.PER_TENSOR), one, None),
                      (Q(aqfq.INT8, aqfq.PER_TENSOR, qmin=-128, qmax=127), one, None),
                      (NV, torch.ones(allb.size // 16), one)]:
        y, c, b = gpu_fwd(sp, x, s, ts)
        y_ref, c_ref, b_ref = oracle_fwd(sp, x, s, ts)
        assert np.array_equal(c, c_ref), f"{sp.fmt}: {np.count_nonzero(c != c_ref)} code mismatches"
        assert np.array_equal(y, y_ref)
    # random scales: v covers arbitrary binary32 values
    xs = x.reshape(1, 60, 1088)
    R, K = xs.shape[1], xs.shape[2]
    for sp, lo, hi in [(Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL), 1e-6, 1e3),
                       (Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127), 1e-6, 1e3)]:
        s = synth.loguniform_f32((R,), lo, hi, seed=40)
        y, c, _ = gpu_fwd(sp, xs, s, None)
        y_ref, c_ref, _ = oracle_fwd(sp, xs, s, None)
        assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref)
    sb = synth.loguniform_f32((xs.numel() // 16,), 1e-6, 1e3, seed=41)
    y, c, b = gpu_fwd(NV, xs, sb, torch.tensor([0.37], dtype=torch.float32))
    y_ref, c_ref, b_ref = oracle_fwd(NV, xs, sb, torch.tensor([0.37], dtype=torch.float32))
    assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref) and np.array_equal(b, b_ref)


def test_empty_and_degenerate_shapes():
    d = dev()
    for B, R, K in [(0, 4, 64), (2, 0, 64), (2, 3, 0)]:
        x = torch.zeros((B, R, K), dtype=torch.bfloat16, device=d)
        y = torch.empty_like(x)
        ts = torch.ones(max(B, 1), device=d)
        sb = torch.ones(max(B * R * K // 16, 1), device=d)
        aqfq.aqfq_qdq_fwd(NV, x, sb, ts, y)
        ch = Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127)
        s = torch.ones(max(B * R, 1), device=d)
        ds = torch.full((max(B * R, 1),), 7.0, device=d)
        aqfq.aqfq_scale_grad(ch, x, x, s, None, dscale=ds)
        torch.cuda.synchronize()
        if B * R > 0:
            assert torch.all(ds[: B * R] == 0)  # empty rows: zero gradient
        tn = Q(aqfq.FP8_E4M3, aqfq.PER_TENSOR)
        dt = torch.full((max(B, 1),), 7.0, device=d)
        wsb = aqfq.aqfq_scale_grad_workspace_bytes(tn, B, R, K)
        ws = torch.empty(max(wsb // 8, 1), dtype=torch.float64, device=d)
        aqfq.aqfq_scale_grad(tn, x, x, torch.ones(max(B, 1), device=d), None, dscale=dt,
                             workspace=ws)
        torch.cuda.synchronize()
        if B > 0:
            assert torch.all(dt[:B] == 0)
    # one block, one row, one batch entry
    case = ("tiny", NV, (1, 1, 16), _x_t, (2e-3, 2e-2), (2e-5, 1e-4))
    x, dy, scale, ts = _inputs(case, seed=50)
    y, c, b = gpu_fwd(NV, x, scale, ts)
    y_ref, c_ref, b_ref = oracle_fwd(NV, x, scale, ts)
    assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref)


def test_per_head_forward_batch_beyond_grid_limit():
    """x [T, H, D] with T above the 65535 grid-y limit: per-head E4M3 QDQ."""
    T, H, D = 70001, 2, 16
    x = synth.head_normal_bf16(T, H, D, 0.1, 10.0, seed=60)
    s = synth.loguniform_f32((H,), 1e-3, 3e-2, seed=61)
    sp = Q(aqfq.FP8_E4M3, aqfq.PER_HEAD)
    y, c, _ = gpu_fwd(sp, x, s, None)
    y_ref, c_ref, _ = oracle_fwd(sp, x, s, None)
    assert np.array_equal(y, y_ref) and np.array_equal(c, c_ref)


@pytest.mark.parametrize("T,H,D,misalign", [(300, 8, 64, False), (97, 5, 48, False),
                                             (1, 3, 16, False), (2048, 32, 128, False),
                                             (301, 7, 24, False), (203, 4, 8, True),
                                             (250, 6, 64, True)])
def test_observer_and_per_head_scale(T, H, D, misalign):
    d = dev()
    x = synth.head_normal_bf16(T, H, D, 0.1, 10.0, seed=70 + T)
    if misalign:  # 16-byte but not 32-byte aligned
        buf = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device=d)
        xd = buf[8:].view(T, H, D)
        xd.copy_(x)
    else:
        xd = x.to(d)
    mn = torch.empty(H, device=d)
    mx = torch.empty(H, device=d)
    aqfq.aqfq_observer_minmax(xd, mn, mx)
    lo, hi = oracle.observer_minmax(bits(x))
    torch.cuda.synchronize()
    assert np.array_equal(mn.cpu().numpy().view(np.uint32), lo.view(np.uint32))
    assert np.array_equal(mx.cpu().numpy().view(np.uint32), hi.view(np.uint32))
    # running merge over token shards equals one pass
    mn2 = torch.empty(H, device=d)
    mx2 = torch.empty(H, device=d)
    cut = max(1, T // 3)
    aqfq.aqfq_observer_minmax(xd[:cut].contiguous(), mn2, mx2)
    aqfq.aqfq_observer_minmax(xd[cut:].contiguous(), mn2, mx2, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(mn2.view(torch.int32), mn.view(torch.int32))
    assert torch.equal(mx2.view(torch.int32), mx.view(torch.int32))
    s = torch.empty(H, device=d)
    aqfq.aqfq_minmax_scale(mn, mx, 448.0, s)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32),
                          oracle.minmax_scale(lo, hi, 448.0).view(np.uint32))


def test_observer_signed_zeros_and_empty():
    d = dev()
    x = torch.zeros((4, 2, 16), dtype=torch.bfloat16)
    xv = x.view(torch.int16)
    xv[1, 0, 3] = -32768  # -0 in head 0 besides +0
    xv[:, 1, :] = -32768  # head 1: only -0
    mn = torch.empty(2, device=d)
    mx = torch.empty(2, device=d)
    aqfq.aqfq_observer_minmax(x.to(d), mn, mx)
    lo, hi = oracle.observer_minmax(bits(x))
    torch.cuda.synchronize()
    assert np.array_equal(mn.cpu().numpy().view(np.uint32), lo.view(np.uint32))
    assert np.array_equal(mx.cpu().numpy().view(np.uint32), hi.view(np.uint32))
    e = torch.empty((0, 2, 16), dtype=torch.bfloat16, device=d)
    aqfq.aqfq_observer_minmax(e, mn, mx)
    torch.cuda.synchronize()
    assert torch.all(mn == float("inf")) and torch.all(mx == float("-inf"))


@pytest.mark.parametrize("misalign", [False, True], ids=["aligned32", "aligned16"])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_scale_init(case, misalign):
    sp = case[1]
    B, R, K = case[2]
    x = case[3](case[2], 80)
    d = dev()
    n = aqfq.scale_numel(sp, B, R, K)
    s = torch.empty(max(n, 1), device=d) if n else None
    ts = torch.empty(B, device=d) if sp.fmt == aqfq.NVFP4 else None
    if misalign:  # 16-byte but not 32-byte aligned
        buf = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device=d)
        xd = buf[8:].view(B, R, K)
        xd.copy_(x)
    else:
        xd = x.to(d)
    aqfq.aqfq_scale_init(sp, xd, s, ts)
    s_ref, ts_ref = oracle.scale_init(ospec(sp), bits(x))
    torch.cuda.synchronize()
    if n:
        assert np.array_equal(s.cpu().numpy()[:n].view(np.uint32), s_ref.view(np.uint32))
    if ts is not None:
        assert np.array_equal(ts.cpu().numpy().view(np.uint32), ts_ref.view(np.uint32))


def test_real_quant_export_layouts():
    """Export (y = NULL) writes the same codes as the full forward, and the
    codes are the deployment tensors: INT4 as pack-quantized int32 words,
    FP8 as float8_e4m3fn, NVFP4 as E2M1 nibbles + E4M3 block scales whose
    product with the tensor scale dequantises to x_hat."""
    d = dev()
    # INT4 g128
    sp = Q(aqfq.INT4, aqfq.PER_GROUP, group=128, qmin=-8, qmax=7)
    x = synth.normal_bf16((2, 24, 256), 0.02, seed=101)
    s = synth.loguniform_f32((2 * 24 * 2,), 2e-3, 2e-2, seed=102)
    y, c, _ = gpu_fwd(sp, x, s, None)
    codes = torch.empty((2, 24, 128), dtype=torch.uint8, device=d)
    aqfq.aqfq_qdq_fwd(sp, x.to(d), s.to(d), None, None, codes)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), c)
    _, c_ref, _ = oracle_fwd(sp, x, s, None)
    words = c_ref.reshape(-1).view(np.uint32)
    nib = c_ref.reshape(-1)
    expect = np.zeros(words.size, np.uint64)
    for i in range(8):  # element 8j+i in bits 4i..4i+3
        el = ((nib[(np.arange(words.size) * 4 + i // 2)] >> (4 * (i % 2))) & 0xF).astype(np.uint64)
        expect |= el << np.uint64(4 * i)
    assert np.array_equal(words.astype(np.uint64), expect)
    # FP8 per channel: codes are float8_e4m3fn values v with x_hat = bf16(v * s)
    sp = Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL)
    x = synth.normal_bf16((1, 16, 128), 0.02, seed=103)
    s = synth.loguniform_f32((16,), 2e-5, 2e-4, seed=104)
    y, c, _ = gpu_fwd(sp, x, s, None)
    v = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).float()
    assert np.array_equal((v * s.view(1, 16, 1)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16), y)
    # NVFP4: e2m1 * e4m3 * g reproduces x_hat
    x = synth.student_t_outliers_bf16((2, 8, 64), 4, 0.02, 5e-3, 20.0, seed=105)
    sb = synth.loguniform_f32((2 * 8 * 4,), 2e-3, 2e-2, seed=106)
    g = synth.loguniform_f32((2,), 2e-5, 1e-4, seed=107)
    y, c, b = gpu_fwd(NV, x, sb, g)
    codes = torch.empty((2, 8, 32), dtype=torch.uint8, device=d)
    blk = torch.empty((2, 8, 4), dtype=torch.uint8, device=d)
    aqfq.aqfq_qdq_fwd(NV, x.to(d), sb.to(d), g.to(d), None, codes, blk)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), c) and np.array_equal(blk.cpu().numpy(), b)
    e2m1 = np.array([oracle.e2m1_decode(k) for k in range(16)])
    lo, hi = e2m1[c & 0xF], e2m1[c >> 4]
    qv = np.stack([lo, hi], -1).reshape(2, 8, 64)
    bs = torch.from_numpy(b.copy()).view(torch.float8_e4m3fn).double().numpy()
    sh = (bs * g.numpy().astype(np.float64).reshape(2, 1, 1)).astype(np.float32).astype(np.float64)
    xh = (qv * np.repeat(sh, 16, axis=-1)).astype(np.float32)
    assert np.array_equal(torch.from_numpy(xh).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16), y)
