"""The five fake-quant workloads as sequences of C-ABI calls on device buffers.

A workload owns its device tensors (seeded synthetic inputs, scales
initialised on the GPU by aqfq_scale_init, outputs) and lists the calls of one
step of its hot path with each call's algorithmic bytes:

  grouped_nvfp4  MoE expert stacks gate_up [128,1536,2048] and down
                 [128,2048,768], Student-t(4)*0.02 with 0.05 % outliers x20:
                 grouped NVFP4 QDQ forward + per-block scale gradient
  nvfp4_wa       NVFP4 weight [4096,4096] (learned block scales) and
                 activations [8192,4096] (dynamic block scales, learned
                 tensor scale, STE input gradient): forward + scale gradients
  int4_fp8       INT4 g128 stack [128,1536,2048] and FP8 per-channel dense
                 [8192,8192]: forward + scale gradients
  observer_fp8   per-head min/max of [65536,32,128] activations, per-head
                 scale, per-head E4M3 QDQ
  int8_channel   INT8 per-channel weight [256,512]: forward + scale gradient
  kd_cakld       distillation loss of student vs teacher logits [4096, 151936]
                 (Qwen3-sized vocabulary), cakld over the whole vocabulary,
                 with the student-logit gradient
  kd_topk        the same with forward KL over the teacher's top-1000 tokens
  *_fused        grouped_nvfp4 / nvfp4_wa / int8_channel with forward and
                 scale gradient of each tensor in one aqfq_qdq_fwd_grad pass
                 (the forward recomputed in the backward pass)

Algorithmic bytes count what the call must move once: inputs read, outputs
written (no codes: the steps do not request them).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable

import torch

from . import aqfq, synth

Q = aqfq.qspec


@dataclass
class Op:
    name: str
    kernel: str
    elems: int
    bytes: int
    run: Callable[[torch.cuda.Stream], None]
    launches: int = 1  # kernels the call launches


@dataclass
class Workload:
    name: str
    description: str
    config: dict
    ops: list = field(default_factory=list)
    inputs: dict = field(default_factory=dict)    # name -> device tensor a user uploads
    outputs: dict = field(default_factory=dict)   # name -> device tensor a user reads back
    # None: the ops run in order on the caller's stream.  Otherwise a list of
    # phases run one after another; a phase is a list of lanes (lists of op
    # indices) that share no data and run concurrently, the first lane on the
    # caller's stream, the others on side streams forked from it and joined
    # back before the next phase.
    phases: list | None = None

    @property
    def bytes_per_step(self) -> int:
        return sum(o.bytes for o in self.ops)

    @property
    def elems_per_step(self) -> int:
        return sum(o.elems for o in self.ops)

    def step(self, stream, hook=None):
        """Launches one step on `stream`.  hook(i, st, end), if given, is called
        on the stream st that runs op i, right before (end False) and right
        after (end True) its launch."""
        def one(i, st):
            if hook is not None:
                hook(i, st, False)
            self.ops[i].run(st)
            if hook is not None:
                hook(i, st, True)

        if not self.phases:
            for i in range(len(self.ops)):
                one(i, stream)
            return
        # every op launches on the stream it is given, so no current-stream
        # switch is needed; lanes fork and join through events
        # (an event may be recorded again once waited on: a wait takes the
        # record made before it)
        side, events = self._lanes(stream.device)
        for phase, (fork, joins) in zip(self.phases, events):
            fork.record(stream)
            for st in side[:len(phase) - 1]:
                st.wait_event(fork)
            for st, lane in zip([stream] + side, phase):
                for i in lane:
                    one(i, st)
            for st, join in zip(side[:len(phase) - 1], joins):
                join.record(st)
                stream.wait_event(join)

    def _lanes(self, device):
        """Side streams and the fork / join events of each phase (made once)."""
        if "_lanes_made" not in self.__dict__:
            n = max(len(ph) for ph in self.phases) - 1
            side = [torch.cuda.Stream(device) for _ in range(n)]
            events = [(torch.cuda.Event(), [torch.cuda.Event() for _ in ph[1:]]) for ph in self.phases]
            self.__dict__["_lanes_made"] = (side, events)
        return self.__dict__["_lanes_made"]

    # ---- end to end with host buffers -------------------------------------------
    def host_buffers(self):
        """Pinned host copies of the inputs (filled from the device) and pinned
        host buffers for the outputs."""
        hin = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in self.inputs.items()}
        for k, v in self.inputs.items():
            hin[k].copy_(v)
        hout = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in self.outputs.items()}
        return hin, hout

    def e2e_step(self, hin, hout, streams):
        """One step from host buffers: upload every input, run the step, download
        every output.  Workloads with slices pipeline upload / compute /
        download over them on three streams."""
        up, comp, down = streams
        slices = getattr(self, "slices", None)
        if not slices:
            with torch.cuda.stream(comp):
                for k, v in self.inputs.items():
                    v.copy_(hin[k], non_blocking=True)
                self.step(comp)
                for k, v in self.outputs.items():
                    hout[k].copy_(v, non_blocking=True)
            return
        # uploads of this step wait for everything queued on the compute stream
        # (the previous step, including its downloads)
        ev_start = torch.cuda.Event()
        ev_start.record(comp)
        up.wait_event(ev_start)
        for sl in slices:
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(up):
                for name, (dev_t, host_t) in sl.inputs(self, hin).items():
                    dev_t.copy_(host_t, non_blocking=True)
                ev_in.record(up)
            ev_done = torch.cuda.Event()
            with torch.cuda.stream(comp):
                comp.wait_event(ev_in)
                for run in sl.ops:
                    run(comp)
                ev_done.record(comp)
            with torch.cuda.stream(down):
                down.wait_event(ev_done)
                for name, (dev_t, host_t) in sl.outputs(self, hout).items():
                    host_t.copy_(dev_t, non_blocking=True)
        # the caller's stream (comp) ends the step after the last download
        ev_end = torch.cuda.Event()
        ev_end.record(down)
        comp.wait_event(ev_end)


def _nvfp4_stack(name, w, dy, dev, ops, inputs, outputs, grouped=True):
    E, N, K = w.shape
    sp = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
    s = torch.empty(E * N * K // 16, device=dev)
    g = torch.empty(E, device=dev)
    aqfq.aqfq_scale_init(sp, w, s, g)
    y = torch.empty_like(w)
    ds = torch.empty_like(s)
    n = w.numel()
    fwd = aqfq.aqfq_grouped_qdq if grouped else aqfq.aqfq_qdq_fwd
    ops.append(Op(f"qdq_fwd {name}", "nvfp4_fwd", n, n * 2 + n // 16 * 4 + n * 2,
                  lambda st: fwd(sp, w, s, g, y, stream=st)))
    ops.append(Op(f"scale_grad {name}", "nvfp4_grad", n, n * 4 + n // 16 * 8,
                  lambda st: aqfq.aqfq_scale_grad(sp, w, dy, s, g, dscale=ds, stream=st)))
    inputs.update({f"{name}": w, f"dy_{name}": dy, f"scale_{name}": s, f"tscale_{name}": g})
    outputs.update({f"y_{name}": y, f"dscale_{name}": ds})
    return sp, s, g


class _ExpertSlice:
    """Experts [e0, e1) of the grouped workload: device/host views of that slice
    of every per-expert tensor and the public calls on them."""

    def __init__(self, wl, e0, e1):
        self.e0, self.e1 = e0, e1
        self.ops = []
        sp = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
        for nm in ("gate_up", "down"):
            x, dy = wl.inputs[nm][e0:e1], wl.inputs[f"dy_{nm}"][e0:e1]
            s, g = self._rows(wl.inputs[f"scale_{nm}"], wl), wl.inputs[f"tscale_{nm}"][e0:e1]
            y, ds = wl.outputs[f"y_{nm}"][e0:e1], self._rows(wl.outputs[f"dscale_{nm}"], wl)
            self.ops.append(lambda st, x=x, s=s, g=g, y=y: aqfq.aqfq_grouped_qdq(sp, x, s, g, y, stream=st))
            self.ops.append(lambda st, x=x, dy=dy, s=s, g=g, ds=ds:
                            aqfq.aqfq_scale_grad(sp, x, dy, s, g, dscale=ds, stream=st))

    def _rows(self, flat, wl):
        E = wl.inputs["gate_up"].shape[0]
        return flat.view(E, -1)[self.e0:self.e1].reshape(-1)

    def _pairs(self, dev, host, wl):
        E = wl.inputs["gate_up"].shape[0]
        return {k: (v.view(E, -1)[self.e0:self.e1], host[k].view(E, -1)[self.e0:self.e1])
                for k, v in dev.items()}

    def inputs(self, wl, hin):
        return self._pairs(wl.inputs, hin, wl)

    def outputs(self, wl, hout):
        return self._pairs(wl.outputs, hout, wl)


# The configuration each workload reports (bench.py's "config"), at its
# default size; builders start from these, so the reference arm can report
# the same dictionary without building device tensors.
CONFIGS = {
    "grouped_nvfp4": {"workload": "grouped_nvfp4_moe_stacks", "gate_up": [128, 1536, 2048],
                      "down": [128, 2048, 768],
                      "format": "nvfp4 (e2m1, 16-elem blocks, e4m3 block scale, fp32 tensor scale)",
                      "values": "student-t(4)*0.02, 0.05% outliers x20",
                      "scale_init": "amax/6, amax/2688"},
    "nvfp4_wa": {"workload": "nvfp4_weight_activation", "w": [4096, 4096], "a": [8192, 4096]},
    "int4_fp8": {"workload": "int4_g128_stack_fp8_channel_dense", "stack": [128, 1536, 2048],
                 "dense": [8192, 8192]},
    "observer_fp8": {"workload": "per_head_observer_fp8", "act": [65536, 32, 128]},
    "head_fp8_learned": {"workload": "per_head_learnable_fp8", "act": [65536, 32, 128]},
    "int8_channel": {"workload": "int8_per_channel_weight", "w": [256, 512]},
    "grouped_nvfp4_gemm": {"workload": "grouped_nvfp4_gemm_gate_up", "x": [65536, 2048],
                           "w": [128, 1536, 2048],
                           "routing": "multinomial, expert popularity exp(N(0,0.3^2))"},
    "grouped_nvfp4_fused": {"workload": "grouped_nvfp4_moe_stacks_fused_fwd_grad",
                            "gate_up": [128, 1536, 2048], "down": [128, 2048, 768],
                            "format": "nvfp4 (e2m1, 16-elem blocks, e4m3 block scale, fp32 tensor scale)",
                            "values": "student-t(4)*0.02, 0.05% outliers x20",
                            "scale_init": "amax/6, amax/2688", "fused": "aqfq_qdq_fwd_grad per stack"},
    "nvfp4_wa_fused": {"workload": "nvfp4_weight_activation_fused_fwd_grad", "w": [4096, 4096],
                       "a": [8192, 4096], "fused": "aqfq_qdq_fwd_grad per tensor"},
    "int8_channel_fused": {"workload": "int8_per_channel_weight_fused_fwd_grad", "w": [256, 512],
                           "fused": "aqfq_qdq_fwd_grad"},
    "kd_cakld": {"workload": "kd_cakld_logits", "logits": [synth.KD_TOKENS, synth.KD_VOCAB],
                 "loss": "cakld", "topk": 0},
    "kd_topk": {"workload": "kd_kl_top1000_logits", "logits": [synth.KD_TOKENS, synth.KD_VOCAB],
                "loss": "kl", "topk": 1000},
}
_KD_RECIPE = ("teacher N(0,4) + one favoured token +U(4,12); student = teacher + N(0,0.09); "
              "10% ignored positions")
for _k in ("kd_cakld", "kd_topk"):
    CONFIGS[_k]["logits_recipe"] = _KD_RECIPE


def grouped_nvfp4(dev, seed=0, experts=None):
    d = synth.cfg3(dev, seed, experts)
    wl = Workload("grouped_nvfp4",
                  "grouped NVFP4 MoE expert stacks gate_up [E,1536,2048] + down [E,2048,768], "
                  "vectorised QDQ fwd + per-block scale grad",
                  dict(CONFIGS["grouped_nvfp4"], gate_up=list(d["gate_up"].shape),
                       down=list(d["down"].shape)))
    for nm in ("gate_up", "down"):
        _nvfp4_stack(nm, d[nm], d[f"dy_{nm}"], dev, wl.ops, wl.inputs, wl.outputs)
    # order: both forwards, then both gradients (forward pass, then backward pass)
    wl.ops = [wl.ops[0], wl.ops[2], wl.ops[1], wl.ops[3]]
    # end to end: 8 slices of experts, upload / compute / download overlapped
    E = d["gate_up"].shape[0]
    n = max(1, min(8, E))
    bounds = [E * i // n for i in range(n + 1)]
    wl.slices = [_ExpertSlice(wl, a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    return wl


def nvfp4_wa(dev, seed=0):
    d = synth.cfg2(dev, seed)
    wl = Workload("nvfp4_wa", "NVFP4 weight [4096,4096] + activations [8192,4096]",
                  dict(CONFIGS["nvfp4_wa"]))
    w = d["w"].unsqueeze(0)
    _nvfp4_stack("w", w, d["dy_w"].unsqueeze(0), dev, wl.ops, wl.inputs, wl.outputs, grouped=False)
    a, dya = d["a"].unsqueeze(0), d["dy_a"].unsqueeze(0)
    spd = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16, mode=aqfq.SCALE_DYNAMIC_BLOCK)
    ga = torch.empty(1, device=dev)
    aqfq.aqfq_scale_init(spd, a, None, ga)
    ya, dxa = torch.empty_like(a), torch.empty_like(a)
    dga = torch.empty(1, device=dev)
    ws = torch.empty(max(1, aqfq.aqfq_scale_grad_workspace_bytes(spd, *a.shape) // 8),
                     dtype=torch.float64, device=dev)
    n = a.numel()
    wl.ops.insert(1, Op("qdq_fwd act", "nvfp4_act_fwd", n, 4 * n,
                        lambda st: aqfq.aqfq_qdq_fwd(spd, a, None, ga, ya, stream=st)))
    wl.ops.append(Op("scale_grad act (+dx)", "nvfp4_act_grad", n, 6 * n,
                     lambda st: aqfq.aqfq_scale_grad(spd, a, dya, None, ga, dtensor_scale=dga,
                                                     dx=dxa, workspace=ws, stream=st), 2))
    wl.inputs.update({"a": a, "dy_a": dya, "tscale_a": ga})
    wl.outputs.update({"y_a": ya, "dx_a": dxa, "dtscale_a": dga})
    # the weight and the activation quantizers share no data: both forwards
    # run concurrently, then both gradients
    wl.phases = [[[0], [1]], [[2], [3]]]
    return wl


def int4_fp8(dev, seed=0):
    d = synth.cfg4(dev, seed)
    wl = Workload("int4_fp8", "INT4 g128 stack [128,1536,2048] + FP8 per-channel [8192,8192]",
                  dict(CONFIGS["int4_fp8"]))
    st4 = Q(aqfq.INT4, aqfq.PER_GROUP, group=128, qmin=-8, qmax=7)
    x4, dy4 = d["stack"], d["dy_stack"]
    s4 = torch.empty(x4.numel() // 128, device=dev)
    aqfq.aqfq_scale_init(st4, x4, s4, None)
    y4, ds4 = torch.empty_like(x4), torch.empty_like(s4)
    n4 = x4.numel()
    sp8 = Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL)
    x8, dy8 = d["dense"].unsqueeze(0), d["dy_dense"].unsqueeze(0)
    s8 = torch.empty(x8.shape[1], device=dev)
    aqfq.aqfq_scale_init(sp8, x8, s8, None)
    y8, ds8 = torch.empty_like(x8), torch.empty_like(s8)
    n8 = x8.numel()
    wl.ops = [
        Op("qdq_fwd int4 stack", "int4_fwd", n4, 4 * n4 + n4 // 128 * 4,
           lambda st: aqfq.aqfq_grouped_qdq(st4, x4, s4, None, y4, stream=st)),
        Op("qdq_fwd fp8 dense", "fp8_fwd", n8, 4 * n8,
           lambda st: aqfq.aqfq_qdq_fwd(sp8, x8, s8, None, y8, stream=st)),
        Op("scale_grad int4 stack", "int4_grad", n4, 4 * n4 + n4 // 128 * 8,
           lambda st: aqfq.aqfq_scale_grad(st4, x4, dy4, s4, None, dscale=ds4, stream=st)),
        Op("scale_grad fp8 dense", "fp8_grad", n8, 4 * n8,
           lambda st: aqfq.aqfq_scale_grad(sp8, x8, dy8, s8, None, dscale=ds8, stream=st)),
    ]
    wl.inputs.update({"stack": x4, "dy_stack": dy4, "scale_stack": s4, "dense": x8,
                      "dy_dense": dy8, "scale_dense": s8})
    wl.outputs.update({"y_stack": y4, "dscale_stack": ds4, "y_dense": y8, "dscale_dense": ds8})
    return wl


def observer_fp8(dev, seed=0):
    d = synth.cfg5(dev, seed)
    x = d["act"]
    T, H, D = x.shape
    wl = Workload("observer_fp8", "per-head observer + E4M3 QDQ on [65536,32,128]",
                  dict(CONFIGS["observer_fp8"], act=[T, H, D]))
    mn, mx, s = (torch.empty(H, device=dev) for _ in range(3))
    y = torch.empty_like(x)
    sp = Q(aqfq.FP8_E4M3, aqfq.PER_HEAD)
    n = x.numel()
    wl.ops = [
        Op("observer_minmax", "observer", n, 2 * n,
           lambda st: aqfq.aqfq_observer_minmax(x, mn, mx, stream=st), 3),
        Op("minmax_scale", "minmax_scale", H, 12 * H,
           lambda st: aqfq.aqfq_minmax_scale(mn, mx, 448.0, s, stream=st)),
        Op("qdq_fwd per-head fp8", "fp8_head_fwd", n, 4 * n,
           lambda st: aqfq.aqfq_qdq_fwd(sp, x, s, None, y, stream=st)),
    ]
    wl.inputs.update({"act": x})
    wl.outputs.update({"y": y, "scale": s})
    return wl


def head_fp8_learned(dev, seed=0):
    """Per-head FP8 E4M3 fake-quant of attention / KV activations with a learnable
    per-head scale: forward, per-head scale gradient and STE input gradient."""
    d = synth.cfg5(dev, seed)
    x = d["act"]
    T, H, D = x.shape
    dy = synth.normal_bf16((T, H, D), 1.0, seed + 1, dev)
    sp = Q(aqfq.FP8_E4M3, aqfq.PER_HEAD)
    s = torch.empty(H, device=dev)
    aqfq.aqfq_scale_init(sp, x, s, None)
    y, dx = torch.empty_like(x), torch.empty_like(x)
    ds = torch.empty(H, device=dev)
    ws = torch.empty(max(1, aqfq.aqfq_scale_grad_workspace_bytes(sp, T, H, D) // 8),
                     dtype=torch.float64, device=dev)
    n = x.numel()
    wl = Workload("head_fp8_learned", "per-head learnable FP8 QDQ on [65536,32,128]: fwd + scale grad + dx",
                  dict(CONFIGS["head_fp8_learned"], act=[T, H, D]))
    wl.ops = [Op("qdq_fwd per-head fp8", "fp8_head_fwd", n, 4 * n,
                 lambda st: aqfq.aqfq_qdq_fwd(sp, x, s, None, y, stream=st)),
              Op("scale_grad per-head fp8 (+dx)", "fp8_head_grad", n, 6 * n,
                 lambda st: aqfq.aqfq_scale_grad(sp, x, dy, s, None, dscale=ds, dx=dx, workspace=ws,
                                                 stream=st), 2)]
    wl.inputs.update({"act": x, "dy": dy, "scale": s})
    wl.outputs.update({"y": y, "dx": dx, "dscale": ds})
    return wl


def int8_channel(dev, seed=0):
    d = synth.cfg1(dev, seed)
    w, dy = d["w"].unsqueeze(0), d["dy"].unsqueeze(0)
    sp = Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127)
    s = torch.empty(w.shape[1], device=dev)
    aqfq.aqfq_scale_init(sp, w, s, None)
    y, ds = torch.empty_like(w), torch.empty_like(s)
    n = w.numel()
    wl = Workload("int8_channel", "INT8 per-channel weight [256,512]",
                  dict(CONFIGS["int8_channel"]))
    wl.ops = [Op("qdq_fwd int8", "int8_fwd", n, 4 * n + 4 * w.shape[1],
                 lambda st: aqfq.aqfq_qdq_fwd(sp, w, s, None, y, stream=st)),
              Op("scale_grad int8", "int8_grad", n, 4 * n + 8 * w.shape[1],
                 lambda st: aqfq.aqfq_scale_grad(sp, w, dy, s, None, dscale=ds, stream=st))]
    wl.inputs.update({"w": w, "dy": dy, "scale": s})
    wl.outputs.update({"y": y, "dscale": ds})
    return wl


def _fused(wl, name, sp, x, dy, s, g, dx=None, ws=None, dyn=False):
    """One aqfq_qdq_fwd_grad call on x: y, the scale gradient (and dx), from one
    read of x and dy.  Returns the outputs."""
    y = torch.empty_like(x)
    n = x.numel()
    ns = 0 if s is None else s.numel()
    if dyn:
        dg = torch.empty_like(g)
        kw = {"dtensor_scale": dg}
        outs = {f"y_{name}": y, f"dtscale_{name}": dg}
    else:
        ds = torch.empty_like(s)
        kw = {"dscale": ds}
        outs = {f"y_{name}": y, f"dscale_{name}": ds}
    if dx is not None:
        outs[f"dx_{name}"] = dx
    nbytes = 6 * n + 8 * ns + (2 * n if dx is not None else 0)  # x, dy, y (+dx); S read, dS written
    wl.ops.append(Op(f"qdq_fwd_grad {name}", "fused_fwd_grad", n, nbytes,
                     lambda st: aqfq.aqfq_qdq_fwd_grad(sp, x, dy, s, g, y, dx=dx, workspace=ws,
                                                       stream=st, **kw),
                     2 if ws is not None else 1))
    wl.outputs.update(outs)


def grouped_nvfp4_fused(dev, seed=0, experts=None):
    """The grouped NVFP4 expert stacks with forward and scale gradient of each
    stack in one pass (aqfq_qdq_fwd_grad): the forward recomputed in the
    backward pass."""
    d = synth.cfg3(dev, seed, experts)
    wl = Workload("grouped_nvfp4_fused",
                  "grouped NVFP4 MoE expert stacks, fused QDQ fwd + per-block scale grad per stack",
                  dict(CONFIGS["grouped_nvfp4_fused"], gate_up=list(d["gate_up"].shape),
                       down=list(d["down"].shape)))
    sp = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
    for nm in ("gate_up", "down"):
        w, dy = d[nm], d[f"dy_{nm}"]
        E, N, K = w.shape
        s = torch.empty(E * N * K // 16, device=dev)
        g = torch.empty(E, device=dev)
        aqfq.aqfq_scale_init(sp, w, s, g)
        _fused(wl, nm, sp, w, dy, s, g)
        wl.inputs.update({nm: w, f"dy_{nm}": dy, f"scale_{nm}": s, f"tscale_{nm}": g})
    return wl


def nvfp4_wa_fused(dev, seed=0):
    """NVFP4 weight [4096,4096] and activations [8192,4096] with forward and
    scale gradient of each tensor in one pass (the activation with its STE
    input gradient)."""
    d = synth.cfg2(dev, seed)
    wl = Workload("nvfp4_wa_fused", "NVFP4 weight + activations, fused fwd + scale grad per tensor",
                  dict(CONFIGS["nvfp4_wa_fused"]))
    sp = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
    w, dyw = d["w"].unsqueeze(0), d["dy_w"].unsqueeze(0)
    s = torch.empty(w.numel() // 16, device=dev)
    g = torch.empty(1, device=dev)
    aqfq.aqfq_scale_init(sp, w, s, g)
    _fused(wl, "w", sp, w, dyw, s, g)
    spd = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16, mode=aqfq.SCALE_DYNAMIC_BLOCK)
    a, dya = d["a"].unsqueeze(0), d["dy_a"].unsqueeze(0)
    ga = torch.empty(1, device=dev)
    aqfq.aqfq_scale_init(spd, a, None, ga)
    ws = torch.empty(max(1, aqfq.aqfq_scale_grad_workspace_bytes(spd, *a.shape) // 8),
                     dtype=torch.float64, device=dev)
    _fused(wl, "a", spd, a, dya, None, ga, dx=torch.empty_like(a), ws=ws, dyn=True)
    wl.inputs.update({"w": w, "dy_w": dyw, "scale_w": s, "tscale_w": g, "a": a, "dy_a": dya,
                      "tscale_a": ga})
    wl.phases = [[[0], [1]]]  # the two tensors' passes run concurrently
    return wl


def int8_channel_fused(dev, seed=0):
    """INT8 per-channel weight [256,512]: forward and scale gradient in one launch."""
    d = synth.cfg1(dev, seed)
    w, dy = d["w"].unsqueeze(0), d["dy"].unsqueeze(0)
    sp = Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127)
    s = torch.empty(w.shape[1], device=dev)
    aqfq.aqfq_scale_init(sp, w, s, None)
    wl = Workload("int8_channel_fused", "INT8 per-channel weight [256,512], fused fwd + scale grad",
                  dict(CONFIGS["int8_channel_fused"]))
    _fused(wl, "w", sp, w, dy, s, None)
    wl.inputs.update({"w": w, "dy": dy, "scale": s})
    return wl


def grouped_nvfp4_gemm(dev, seed=0, tokens=8192, topk=8, experts=None):
    """MoE gate_up projection with NVFP4 fake-quantized expert weights (nvfp4a16):
    routed activations X [tokens * topk, 2048] grouped by expert, W [128, 1536, 2048].
    Fused: one aqfq_grouped_qdq_gemm call.  Unfused reference path: the stack's
    QDQ (aqfq_grouped_qdq, w_hat written to HBM) then one cuBLAS GEMM per expert."""
    E, N, K = synth.CFG3_GATE_UP
    if experts is not None:  # smaller profiling case: fewer experts, same tokens per expert
        tokens = tokens * experts // E
        E = experts
    M = tokens * topk
    counts = synth.routing_counts(E, M, seed + 7)
    off = torch.zeros(E + 1, dtype=torch.int32)
    off[1:] = torch.cumsum(counts, 0).to(torch.int32)
    offd = off.to(dev)
    w = synth.student_t_outliers_bf16((E, N, K), 4, 0.02, 5e-4, 20.0, seed, dev)
    x = synth.normal_bf16((M, K), 1.0, seed + 1, dev)
    sp = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
    s = torch.empty(E * N * K // 16, device=dev)
    g = torch.empty(E, device=dev)
    aqfq.aqfq_scale_init(sp, w, s, g)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    y2 = torch.empty_like(y)
    wh = torch.empty_like(w)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flops = 2 * M * N * K
    bounds = [int(v) for v in off]

    def unfused(st):
        aqfq.aqfq_grouped_qdq(sp, w, s, g, wh, stream=st)
        for e in range(E):
            lo, hi = bounds[e], bounds[e + 1]
            if hi > lo:
                torch.matmul(x[lo:hi], wh[e].t(), out=y2[lo:hi])

    wl = Workload("grouped_nvfp4_gemm",
                  "fused NVFP4 weight fake-quant + grouped GEMM, X [65536,2048] x W [128,1536,2048]",
                  dict(CONFIGS["grouped_nvfp4_gemm"], x=[M, K], w=[E, N, K]))
    wl.ops = [Op("fused qdq+grouped gemm", "qdq_gemm", M * N, flops,
                 lambda st: aqfq.aqfq_grouped_qdq_gemm(x, offd, w, s, g, y, err, stream=st))]
    wl.reference_ops = [Op("unfused: qdq stack + per-expert cuBLAS", "qdq_then_cublas", M * N, flops,
                           unfused, 1)]
    wl.flops = flops
    wl.inputs.update({"x": x, "w": w, "scale": s, "tscale": g, "m_offsets": offd})
    wl.outputs.update({"y": y})
    wl.err = err
    return wl


def _kd(name, kd_type, topk, dev, seed=0, T=synth.KD_TOKENS, V=synth.KD_VOCAB):
    """Distillation loss + student-logit gradient for T positions over a
    V-token vocabulary (one aqfq_kd_loss call: count, loss and mean kernels).
    Unfused reference path: the same loss in eager torch (fp32 log-softmax,
    autograd for the gradient)."""
    student, teacher, labels = synth.kd_logits(T, V, seed, dev)
    losses = torch.empty(3, device=dev)
    ds = torch.empty_like(student)
    ws = torch.empty(aqfq.aqfq_kd_workspace_bytes(T), dtype=torch.uint8, device=dev)
    n = T * V
    label = {aqfq.KD_CAKLD: "cakld", aqfq.KD_KL: "kl", aqfq.KD_RKL: "rkl", aqfq.KD_MSE: "mse"}[kd_type]
    wl = Workload(name, f"distillation loss {label}{f' top-{topk}' if topk else ''}, logits [{T}, {V}]",
                  dict(CONFIGS[name], logits=[T, V]))
    # algorithmic bytes: at each valid position both logit rows read and the
    # gradient row written (top-K: the teacher row, the student's K support
    # values and the gradient row); only the (zero) gradient row at an
    # ignored one; the labels
    n_valid = int(((labels >= 0) & (labels < V)).sum())
    per_valid = (4 * V + 2 * topk) if topk else 6 * V
    nbytes = per_valid * n_valid + 2 * (T - n_valid) * V + 4 * T
    wl.ops = [Op(f"kd_loss {label}", "kd_loss", n, nbytes,
                 lambda st: aqfq.aqfq_kd_loss(kd_type, student, teacher, labels, losses, ws, topk=topk,
                                              dstudent=ds, stream=st), launches=3)]

    def eager(st):
        with torch.cuda.stream(st), torch.enable_grad():
            sv = student.float().requires_grad_(True)
            tv = teacher.float()
            keep = (labels >= 0) & (labels < V)
            idx = torch.nonzero(keep).squeeze(1)
            a, b = tv[idx], sv[idx]
            if topk:
                sup = torch.topk(a, topk, dim=-1).indices
                a, b = a.gather(1, sup), b.gather(1, sup)
            lpt, lps = torch.log_softmax(a, -1), torch.log_softmax(b, -1)
            fkl = (lpt.exp() * (lpt - lps)).sum(-1)
            if kd_type == aqfq.KD_CAKLD:
                rkl = (lps.exp() * (lps - lpt)).sum(-1)
                conf = torch.softmax(tv[idx], -1).gather(1, labels[idx].long()[:, None]).squeeze(1)
                loss = (conf * rkl + (1 - conf) * fkl).mean()
            else:
                loss = fkl.mean()
            loss.backward()
            ds.copy_(sv.grad)

    wl.reference_ops = [Op("unfused: eager torch fp32 + autograd", "torch_eager", n, nbytes, eager)]
    wl.inputs.update({"student": student, "teacher": teacher, "labels": labels})
    wl.outputs.update({"losses": losses, "dstudent": ds})
    return wl


def kd_cakld(dev, seed=0, tokens=synth.KD_TOKENS):
    return _kd("kd_cakld", aqfq.KD_CAKLD, 0, dev, seed, T=tokens)


def kd_topk(dev, seed=0, tokens=synth.KD_TOKENS):
    return _kd("kd_topk", aqfq.KD_KL, 1000, dev, seed, T=tokens)


BUILDERS = {"grouped_nvfp4": grouped_nvfp4, "grouped_nvfp4_fused": grouped_nvfp4_fused,
            "nvfp4_wa_fused": nvfp4_wa_fused, "int8_channel_fused": int8_channel_fused,
            "nvfp4_wa": nvfp4_wa, "int4_fp8": int4_fp8,
            "observer_fp8": observer_fp8, "int8_channel": int8_channel,
            "head_fp8_learned": head_fp8_learned, "grouped_nvfp4_gemm": grouped_nvfp4_gemm,
            "kd_cakld": kd_cakld, "kd_topk": kd_topk}
