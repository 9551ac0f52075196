"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (the same workload objects and C-ABI calls).  The GPU runs every call on
the whole tensors; the oracle recomputes complete units the CPU finishes in
seconds: whole experts of the stacks, whole weight / activation tensors where
they are small enough, sampled rows of the dense FP8 weight (its units are
rows), the whole observer.  The oracle initialises its own scales from the
same data; they must equal the GPU's scale init bit for bit before the
forward and gradient are compared."""
import gc

import numpy as np
import pytest
import torch

import oracle
from learnable_scale_fake_gb300 import synth, workloads
from paritylib import assert_grad_close, bits, dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
O = oracle


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _run(wl):
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        wl.step(st)
    torch.cuda.synchronize()


def _f32(t):
    return t.detach().cpu().numpy()


def _check_block(osp, x, dy, s_gpu, ts_gpu, y_gpu, ds_gpu, dts_gpu=None, dx_gpu=None):
    """x, dy: [B, R, K] host BF16 bits of complete units; *_gpu: the GPU results
    for the same units (numpy)."""
    s, ts = O.scale_init(osp, x)
    if s is not None:
        assert np.array_equal(s.view(np.uint32), np.asarray(s_gpu, np.float32).reshape(-1).view(np.uint32)), \
            "scale init differs"
    if ts is not None:
        assert np.array_equal(ts.view(np.uint32), np.asarray(ts_gpu, np.float32).reshape(-1).view(np.uint32)), \
            "tensor-scale init differs"
    y, _, _ = O.qdq_fwd(osp, x, s, ts)
    assert np.array_equal(y, y_gpu), f"{np.count_nonzero(y != y_gpu)} x_hat mismatches"
    g = O.scale_grad(osp, x, dy, s, ts)
    if ds_gpu is not None:
        assert_grad_close(np.asarray(ds_gpu).reshape(-1), g["dscale"], g["dscale_abs"])
    if dts_gpu is not None:
        assert_grad_close(np.asarray(dts_gpu).reshape(-1), g["dtensor_scale"], g["dtensor_scale_abs"],
                          what="dtensor_scale")
    if dx_gpu is not None:
        assert np.array_equal(g["dx"], dx_gpu)


def test_grouped_nvfp4_stacks_full_size():
    wl = workloads.grouped_nvfp4(dev())
    _run(wl)
    osp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    for nm, experts in (("gate_up", (0, 77, 127)), ("down", (0, 127))):
        x = wl.inputs[nm]
        E, N, K = x.shape
        nb = N * K // 16
        for e in experts:
            xs = bits(x[e:e + 1])
            _check_block(osp, xs, bits(wl.inputs[f"dy_{nm}"][e:e + 1]),
                         _f32(wl.inputs[f"scale_{nm}"][e * nb:(e + 1) * nb]),
                         _f32(wl.inputs[f"tscale_{nm}"][e:e + 1]),
                         bits(wl.outputs[f"y_{nm}"][e:e + 1]),
                         _f32(wl.outputs[f"dscale_{nm}"][e * nb:(e + 1) * nb]))


def test_nvfp4_weight_and_activation_full_size():
    wl = workloads.nvfp4_wa(dev())
    _run(wl)
    osp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    _check_block(osp, bits(wl.inputs["w"]), bits(wl.inputs["dy_w"]), _f32(wl.inputs["scale_w"]),
                 _f32(wl.inputs["tscale_w"]), bits(wl.outputs["y_w"]), _f32(wl.outputs["dscale_w"]))
    osd = O.spec(O.NVFP4, O.PER_GROUP, group=16, mode=O.SCALE_DYNAMIC_BLOCK)
    _check_block(osd, bits(wl.inputs["a"]), bits(wl.inputs["dy_a"]), None, _f32(wl.inputs["tscale_a"]),
                 bits(wl.outputs["y_a"]), None, dts_gpu=_f32(wl.outputs["dtscale_a"]),
                 dx_gpu=bits(wl.outputs["dx_a"]))


def test_int4_stack_and_fp8_dense_full_size():
    wl = workloads.int4_fp8(dev())
    _run(wl)
    osp = O.spec(O.INT4, O.PER_GROUP, group=128, qmin=-8, qmax=7)
    x = wl.inputs["stack"]
    E, N, K = x.shape
    ng = N * K // 128
    for e in (0, 64, 127):
        _check_block(osp, bits(x[e:e + 1]), bits(wl.inputs["dy_stack"][e:e + 1]),
                     _f32(wl.inputs["scale_stack"][e * ng:(e + 1) * ng]), None,
                     bits(wl.outputs["y_stack"][e:e + 1]),
                     _f32(wl.outputs["dscale_stack"][e * ng:(e + 1) * ng]))
    osp = O.spec(O.FP8_E4M3, O.PER_CHANNEL)
    for r0 in (0, 4000, 8128):
        rows = slice(r0, r0 + 64)
        _check_block(osp, bits(wl.inputs["dense"][:, rows]), bits(wl.inputs["dy_dense"][:, rows]),
                     _f32(wl.inputs["scale_dense"][rows]), None, bits(wl.outputs["y_dense"][:, rows]),
                     _f32(wl.outputs["dscale_dense"][rows]))


def test_per_head_observer_and_fp8_full_size():
    wl = workloads.observer_fp8(dev())
    _run(wl)
    x = wl.inputs["act"]
    lo, hi = O.observer_minmax(bits(x))
    s = O.minmax_scale(lo, hi, 448.0)
    assert np.array_equal(s.view(np.uint32), _f32(wl.outputs["scale"]).view(np.uint32))
    osp = O.spec(O.FP8_E4M3, O.PER_HEAD)
    for t0 in (0, 65536 - 256):
        y, _, _ = O.qdq_fwd(osp, bits(x[t0:t0 + 256]), s)
        assert np.array_equal(y, bits(wl.outputs["y"][t0:t0 + 256]))


def test_int8_channel_full_size():
    wl = workloads.int8_channel(dev())
    _run(wl)
    osp = O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127)
    _check_block(osp, bits(wl.inputs["w"]), bits(wl.inputs["dy"]), _f32(wl.inputs["scale"]), None,
                 bits(wl.outputs["y"]), _f32(wl.outputs["dscale"]))


def test_grouped_e2e_pipeline_matches_device_step():
    """The host-buffer path (uploads / compute / downloads overlapped over
    expert slices on three streams) returns the same outputs as the device
    step, on two steps in a row."""
    d = dev()
    wl = workloads.grouped_nvfp4(d, experts=16)
    _run(wl)
    ref = {k: v.clone() for k, v in wl.outputs.items()}
    hin, hout = wl.host_buffers()
    for v in wl.outputs.values():
        v.zero_()
    streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
    for _ in range(2):
        for v in hout.values():
            v.zero_()
        wl.e2e_step(hin, hout, streams)
        torch.cuda.synchronize()
        for k, v in ref.items():
            assert torch.equal(hout[k].view(torch.uint8), v.cpu().view(torch.uint8)), k


def test_fused_gemm_full_size_sampled():
    """The fused fake-quant + grouped GEMM on the bench's workload (65536 routed
    rows, W [128, 1536, 2048], uneven routing): outputs at every expert's first
    and last row, on both sides of every 512-row group boundary and at random
    rows, three columns each, recomputed by the oracle from the one X row and
    the weight rows they need; within the same bound as the small cases
    (|y - ref| <= 2^-8 |ref| + K 2^-24 sum_k |x w_hat|)."""
    d = dev()
    wl = workloads.grouped_nvfp4_gemm(d)
    _run(wl)
    assert int(wl.err.item()) == 0, "a pipeline wait timed out"
    x, off, w = wl.inputs["x"], wl.inputs["m_offsets"], wl.inputs["w"]
    s, g, y = wl.inputs["scale"], wl.inputs["tscale"], wl.outputs["y"]
    E, N, K = w.shape
    offs = off.cpu().numpy().astype(np.int64)
    rows = set()
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            rows.update((lo, hi - 1))
        for b in range(lo + 512, hi, 512):  # a group boundary: last row before, first after
            rows.update((b - 1, b))
    rng = np.random.default_rng(5)
    rows.update(int(r) for r in rng.integers(0, x.shape[0], 64))
    rows = np.array(sorted(rows), dtype=np.int64)
    assert rows.size > 3 * E  # the routing is uneven: many experts span two groups
    cols = rng.integers(0, N, (rows.size, 3))
    cols[0, 0], cols[-1, -1] = 0, N - 1
    xr = bits(x[torch.from_numpy(rows).to(d)].cpu())
    sv = s.view(E, N, K // 16)
    gh = _f32(g)
    for i, m in enumerate(rows):
        e = int(np.searchsorted(offs, m, side="right") - 1)
        c = torch.from_numpy(cols[i]).to(d)
        ref, absref = O.grouped_qdq_gemm(xr[i:i + 1], [0, 1], bits(w[e, c].cpu())[None],
                                         _f32(sv[e, c]).reshape(-1), gh[e:e + 1])
        got = y[int(m), c].float().cpu().numpy().astype(np.float64)
        tol = 2.0 ** -8 * np.abs(ref[0]) + K * 2.0 ** -24 * absref[0]
        assert np.all(np.abs(got - ref[0]) <= tol), (int(m), e, cols[i], got, ref[0])
