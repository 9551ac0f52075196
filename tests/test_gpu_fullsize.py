"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (the same workload objects and C-ABI calls), element by element over
every unit: the GPU runs every call on the whole tensors and the oracle
recomputes all of them (every expert of both NVFP4 stacks, the whole INT4
stack, every row of the dense FP8 weight, every token of the per-head QDQ,
every output of the fused GEMM).  The oracle initialises its own scales from
the same data; they must equal the GPU's scale init bit for bit before the
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
    # the workload's set-up (inputs, scale init) ran on the current stream
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
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
    """All 128 experts of gate_up [128,1536,2048] and down [128,2048,768]:
    x_hat bit-exact, every block-scale gradient within the tolerance."""
    wl = workloads.grouped_nvfp4(dev())
    _run(wl)
    osp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    for nm in ("gate_up", "down"):
        _check_block(osp, bits(wl.inputs[nm]), bits(wl.inputs[f"dy_{nm}"]),
                     _f32(wl.inputs[f"scale_{nm}"]), _f32(wl.inputs[f"tscale_{nm}"]),
                     bits(wl.outputs[f"y_{nm}"]), _f32(wl.outputs[f"dscale_{nm}"]))
        gc.collect()


def test_fused_workloads_full_size():
    """The fused forward + gradient workloads (one aqfq_qdq_fwd_grad pass per
    tensor) at the bench's sizes: every expert of both NVFP4 stacks, the NVFP4
    weight and activation tensors (with dx), the INT8 per-channel weight."""
    osp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    wl = workloads.grouped_nvfp4_fused(dev())
    _run(wl)
    for nm in ("gate_up", "down"):
        _check_block(osp, bits(wl.inputs[nm]), bits(wl.inputs[f"dy_{nm}"]),
                     _f32(wl.inputs[f"scale_{nm}"]), _f32(wl.inputs[f"tscale_{nm}"]),
                     bits(wl.outputs[f"y_{nm}"]), _f32(wl.outputs[f"dscale_{nm}"]))
        gc.collect()
    del wl
    gc.collect()
    wl = workloads.nvfp4_wa_fused(dev())
    _run(wl)
    _check_block(osp, bits(wl.inputs["w"]), bits(wl.inputs["dy_w"]), _f32(wl.inputs["scale_w"]),
                 _f32(wl.inputs["tscale_w"]), bits(wl.outputs["y_w"]), _f32(wl.outputs["dscale_w"]))
    osd = O.spec(O.NVFP4, O.PER_GROUP, group=16, mode=O.SCALE_DYNAMIC_BLOCK)
    _check_block(osd, bits(wl.inputs["a"]), bits(wl.inputs["dy_a"]), None, _f32(wl.inputs["tscale_a"]),
                 bits(wl.outputs["y_a"]), None, dts_gpu=_f32(wl.outputs["dtscale_a"]),
                 dx_gpu=bits(wl.outputs["dx_a"]))
    wl = workloads.int8_channel_fused(dev())
    _run(wl)
    _check_block(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), bits(wl.inputs["w"]),
                 bits(wl.inputs["dy"]), _f32(wl.inputs["scale"]), None, bits(wl.outputs["y_w"]),
                 _f32(wl.outputs["dscale_w"]))


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
    """The whole INT4 g128 stack [128,1536,2048] and every row of the FP8
    per-channel dense weight [8192,8192]."""
    wl = workloads.int4_fp8(dev())
    _run(wl)
    osp = O.spec(O.INT4, O.PER_GROUP, group=128, qmin=-8, qmax=7)
    _check_block(osp, bits(wl.inputs["stack"]), bits(wl.inputs["dy_stack"]),
                 _f32(wl.inputs["scale_stack"]), None, bits(wl.outputs["y_stack"]),
                 _f32(wl.outputs["dscale_stack"]))
    gc.collect()
    osp = O.spec(O.FP8_E4M3, O.PER_CHANNEL)
    _check_block(osp, bits(wl.inputs["dense"]), bits(wl.inputs["dy_dense"]),
                 _f32(wl.inputs["scale_dense"]), None, bits(wl.outputs["y_dense"]),
                 _f32(wl.outputs["dscale_dense"]))


def test_per_head_observer_and_fp8_full_size():
    """Observer min/max and the per-head scale bit-exact, then the per-head
    E4M3 QDQ of all 65536 tokens x 32 heads x 128."""
    wl = workloads.observer_fp8(dev())
    _run(wl)
    x = bits(wl.inputs["act"])
    lo, hi = O.observer_minmax(x)
    s = O.minmax_scale(lo, hi, 448.0)
    assert np.array_equal(s.view(np.uint32), _f32(wl.outputs["scale"]).view(np.uint32))
    osp = O.spec(O.FP8_E4M3, O.PER_HEAD)
    y, _, _ = O.qdq_fwd(osp, x, s)
    got = bits(wl.outputs["y"])
    assert np.array_equal(y, got), f"{np.count_nonzero(y != got)} x_hat mismatches"


def test_per_head_learnable_fp8_full_size():
    """The per-head learnable-scale workload [65536,32,128]: forward, per-head
    scale gradient and STE input gradient over every token."""
    wl = workloads.head_fp8_learned(dev())
    _run(wl)
    osp = O.spec(O.FP8_E4M3, O.PER_HEAD)
    _check_block(osp, bits(wl.inputs["act"]), bits(wl.inputs["dy"]), _f32(wl.inputs["scale"]), None,
                 bits(wl.outputs["y"]), _f32(wl.outputs["dscale"]), dx_gpu=bits(wl.outputs["dx"]))


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


def test_fused_gemm_full_size():
    """The fused fake-quant + grouped GEMM on the bench's workload (65536 routed
    rows, W [128, 1536, 2048], uneven routing): every output against the
    oracle's double GEMM of its own x_hat, within
    |y - ref| <= 2^-8 |ref| + K 2^-24 sum_k |x w_hat|
    (the rounding of y to BF16, 8 significant bits, plus FP32 accumulation
    over K in the tensor cores' order)."""
    d = dev()
    wl = workloads.grouped_nvfp4_gemm(d)
    _run(wl)
    assert int(wl.err.item()) == 0, "a pipeline wait timed out"
    x, off, w = wl.inputs["x"], wl.inputs["m_offsets"], wl.inputs["w"]
    s, g, y = wl.inputs["scale"], wl.inputs["tscale"], wl.outputs["y"]
    E, N, K = w.shape
    offs = off.cpu().numpy().astype(np.int64)
    ref, absref = O.grouped_qdq_gemm(bits(x), offs, bits(w), _f32(s), _f32(g))
    got = y.float().cpu().numpy().astype(np.float64)
    m = int(offs[-1])
    tol = 2.0 ** -8 * np.abs(ref[:m]) + K * 2.0 ** -24 * absref[:m]
    bad = np.argwhere(np.abs(got[:m] - ref[:m]) > tol)
    assert bad.size == 0, (f"{len(bad)} outputs beyond the bound, e.g. row {bad[0][0]} col {bad[0][1]}: "
                           f"{got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}")
