"""Benchmark of the fake-quant hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload grouped_nvfp4|nvfp4_wa|int4_fp8|observer_fp8|int8_channel|
                                head_fp8_learned|grouped_nvfp4_fused|nvfp4_wa_fused|
                                int8_channel_fused|grouped_nvfp4_gemm|kd_cakld|kd_topk]

One step = one pass of the workload's whole hot path: for the default
workload (grouped NVFP4 MoE expert stacks, gate_up [128,1536,2048] + down
[128,2048,768]) the vectorised QDQ forward of both stacks and the per-block
scale gradient of both stacks, through the C ABI.  Inputs are resident in
HBM and larger than L2.  Prints one JSON line (rank 0).

Metric: algorithmic HBM bytes moved per second (GB/s), with elements/s and
the fraction of the measured HBM copy bandwidth.  Under torchrun each rank
runs the same workload on its own GPU (independent replicas, weak scaling);
the time is the max over ranks.

--impl reference times the CPU oracle (the plain double-precision
implementation) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="grouped_nvfp4")
    ap.add_argument("--experts", type=int, default=None,
                    help="grouped_nvfp4 only: truncate the expert axis (small profiling case)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="kd_cakld / kd_topk only: number of positions (small profiling case)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay leg")
    return ap.parse_args()


# ---------------------------------------------------------------------------------------
# peaks, clocks, profile summaries
# ---------------------------------------------------------------------------------------

def tensor_peak():
    """Measured dense BF16 tensor throughput (burst: the kernel is timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(files):
    """Hash of the named CUDA sources (paths relative to the repository): a
    stored ncu traffic figure is valid only for the sources it was taken on."""
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(os.path.basename(f).encode() + fh.read())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def stored_traffic(op_name):
    """DRAM bytes per launch of op `op_name` from the stored ncu capture
    (profiles/traffic.json: op -> bytes, sources, their digest), if it was
    taken on the current state of the sources it names; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            row = json.load(f)["ops"].get(op_name)
    except (OSError, ValueError, KeyError, AttributeError):
        return None
    if not row:
        return None
    try:
        if row["sources"] and row["digest"] == source_digest(row["sources"]):
            return int(row["dram_bytes_per_launch"])
    except (OSError, KeyError, TypeError, ValueError):
        return None
    return None


def rank_plan(gpus, env):
    """How this process serves `--gpus N`: "run" (a single process with N = 1,
    or one rank of an N-rank launch), "spawn" (N > 1 outside a launcher: start
    N ranks on this node), or an error message when the launcher's world size
    disagrees with N."""
    world = env.get("WORLD_SIZE")
    if gpus < 1:
        return "error: --gpus must be at least 1"
    if world is None:
        return "run" if gpus == 1 else "spawn"
    if int(world) != gpus:
        return f"error: --gpus {gpus} but the launcher started WORLD_SIZE={world} ranks"
    return "run"


def spawn_ranks(gpus, argv):
    """Runs this script as `gpus` ranks of one node (torch.distributed.run,
    rendezvous on 127.0.0.1) and returns the launcher's exit code."""
    import socket

    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self, t_begin, t_end):
        """Samples whose timestamp lies in [t_begin, t_end] (host wall clock,
        seconds); if the region was shorter than the sampling period, the
        sample closest to the region's middle."""
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        raw = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 7]
        os.unlink(self.file.name)
        rows = []
        for r in raw:
            try:
                ts = time.mktime(time.strptime(r[0].strip()[:19], "%Y/%m/%d %H:%M:%S"))
                ts += float("0" + r[0].strip()[19:]) if "." in r[0] else 0.0
                rows.append((ts, [c.strip() for c in r[1:]]))
            except ValueError:
                continue
        inside = [r for t, r in rows if t_begin <= t <= t_end]
        if not inside and rows:
            mid = 0.5 * (t_begin + t_end)
            inside = [min(rows, key=lambda tr: abs(tr[0] - mid))[1]]
        if not inside:
            return {"samples": 0}
        sm = [float(r[0]) for r in inside if r[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3 + i] == "Active"})
        try:
            smax = float(inside[0][1])
        except ValueError:
            smax = None
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------------------
# CPU oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------------------

def _oracle_jobs(name, inputs):
    """(label, x, dy, oracle spec, algorithmic bytes per element of fwd + grad)
    for the workload's tensors; x / dy are [units, ...] so that a sample is a
    leading slice.  The bytes per element match the workload's GPU ops."""
    import oracle as O

    def flat(t):
        return t.reshape(-1, t.shape[-1])

    if name in ("grouped_nvfp4", "grouped_nvfp4_fused"):
        sp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
        bpe = 8.75 if name == "grouped_nvfp4" else 6.5  # separate calls / one pass per stack
        return [(nm, inputs[nm], inputs[f"dy_{nm}"], sp, bpe) for nm in ("gate_up", "down")], "experts"
    if name == "int4_fp8":
        return [("stack", inputs["stack"], inputs["dy_stack"],
                 O.spec(O.INT4, O.PER_GROUP, group=128, qmin=-8, qmax=7), 4.03125 + 4.0625),
                ("dense", flat(inputs["dense"]).reshape(-1, 64, 8192),
                 flat(inputs["dy_dense"]).reshape(-1, 64, 8192),
                 O.spec(O.FP8_E4M3, O.PER_CHANNEL), 8.0)], "leading units (expert / 64 rows)"
    if name in ("nvfp4_wa", "nvfp4_wa_fused"):
        fused = name == "nvfp4_wa_fused"
        return [("w", flat(inputs["w"]).reshape(-1, 64, 4096), flat(inputs["dy_w"]).reshape(-1, 64, 4096),
                 O.spec(O.NVFP4, O.PER_GROUP, group=16), 6.5 if fused else 8.75),
                ("a", flat(inputs["a"]).reshape(-1, 64, 4096), flat(inputs["dy_a"]).reshape(-1, 64, 4096),
                 O.spec(O.NVFP4, O.PER_GROUP, group=16, mode=O.SCALE_DYNAMIC_BLOCK),
                 8.0 if fused else 10.0)], "leading units of 64 rows"
    if name in ("int8_channel", "int8_channel_fused"):
        return [("w", flat(inputs["w"]).reshape(-1, 16, 512), flat(inputs["dy"]).reshape(-1, 16, 512),
                 O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127),
                 6.0 if name == "int8_channel_fused" else 8.0)], "leading units of 16 rows"
    if name == "grouped_nvfp4_gemm":
        return [("gemm", inputs["w"], None, "gemm", 0.0)], "experts (with their routed rows)"
    if name in ("kd_cakld", "kd_topk"):
        kt, k = (O.KD_CAKLD, 0) if name == "kd_cakld" else (O.KD_KL, 1000)
        return [("kd", inputs["teacher"], inputs["student"], ("kd", kt, k, inputs["labels"]), 6.0)], \
            "leading positions"
    if name == "head_fp8_learned":
        return [("act", inputs["act"], inputs["dy"], O.spec(O.FP8_E4M3, O.PER_HEAD), 10.0)], \
            "leading tokens"
    return [("act", inputs["act"], None, None, 6.0)], "leading tokens"


def oracle_run(name, inputs, k):
    """The oracle, as it stands, on the first k units of each tensor (forward +
    scale gradient; observer + scale + per-head QDQ for the observer workload).
    Returns (algorithmic bytes, elements, seconds)."""
    import oracle as O
    from learnable_scale_fake_gb300 import synth

    jobs, _ = _oracle_jobs(name, inputs)
    nbytes = elems = 0
    secs = 0.0
    for nm, x, dy, sp, bpe in jobs:
        kk = min(k, x.shape[0])
        if sp == "gemm":  # fused fake-quant GEMM: the first kk experts and their rows
            off = [int(v) for v in inputs["m_offsets"][: kk + 1]]
            xs = synth.bf16_bits(inputs["x"][: off[-1]])
            w = synth.bf16_bits(inputs["w"][:kk])
            sc, ts = O.scale_init(O.spec(O.NVFP4, O.PER_GROUP, group=16), w)
            t0 = time.perf_counter()
            O.grouped_qdq_gemm(xs, off, w, sc, ts)
            secs += time.perf_counter() - t0
            nbytes += 2 * off[-1] * w.shape[1] * w.shape[2]  # FLOPs
            elems += off[-1] * w.shape[1]
            continue
        if isinstance(sp, tuple) and sp[0] == "kd":  # distillation loss: the first kk positions
            _, kt, topk, labels = sp
            tb, sb = synth.bf16_bits(x[:kk]), synth.bf16_bits(dy[:kk])
            lab = labels[:kk].cpu().numpy()
            t0 = time.perf_counter()
            O.kd_loss(kt, sb, tb, lab, topk=topk)
            secs += time.perf_counter() - t0
            # the workload's algorithmic bytes for these positions: both rows
            # and the gradient row (top-K: the teacher row, K student values
            # and the gradient row) per valid position, the zero gradient row
            # per ignored one, the labels
            V = tb.shape[1]
            n_valid = int(((lab >= 0) & (lab < V)).sum())
            per_valid = (4 * V + 2 * topk) if topk else 6 * V
            nbytes += per_valid * n_valid + 2 * V * (kk - n_valid) + 4 * kk
            elems += tb.size
            continue
        xb = synth.bf16_bits(x[:kk])
        if sp is None:  # observer + scale + per-head E4M3 QDQ
            t0 = time.perf_counter()
            lo, hi = O.observer_minmax(xb)
            sc = O.minmax_scale(lo, hi, 448.0)
            O.qdq_fwd(O.spec(O.FP8_E4M3, O.PER_HEAD), xb, sc)
            secs += time.perf_counter() - t0
            nbytes += int(bpe * xb.size)
            elems += 2 * xb.size
            continue
        db = synth.bf16_bits(dy[:kk])
        if xb.ndim == 2:
            xb, db = xb[None], db[None]
        s, ts = O.scale_init(sp, xb)  # the oracle's own scale init, untimed
        t0 = time.perf_counter()
        O.qdq_fwd(sp, xb, s, ts)
        O.scale_grad(sp, xb, db, s, ts)
        secs += time.perf_counter() - t0
        m = xb.size
        elems += 2 * m
        nbytes += int(m * bpe)
    return int(nbytes), elems, secs


def oracle_pick(name, inputs, target_s):
    """Grows the sample (x2) until one oracle pass takes at least target_s / 2
    (so a pass lasts about target_s / 2 .. target_s), or the inputs run out."""
    jobs, unit = _oracle_jobs(name, inputs)
    limit = min(j[1].shape[0] for j in jobs)
    k = 1
    while True:
        res = oracle_run(name, inputs, k)
        if res[2] >= target_s / 2 or k >= limit:
            return k, res, f"first {k} {unit} of each tensor"
        k = min(limit, max(k + 1, int(k * min(4.0, 0.75 * target_s / max(res[2], 1e-3)))))


def _gemm_sample_inputs(experts=4):
    """CPU inputs for the oracle leg of the fused GEMM workload: the first
    experts of the routed problem (same shapes and distributions)."""
    import torch

    from learnable_scale_fake_gb300 import synth

    E, N, K = synth.CFG3_GATE_UP
    counts = synth.routing_counts(E, 8192 * 8, 7)[:experts]
    off = torch.zeros(experts + 1, dtype=torch.int64)
    off[1:] = torch.cumsum(counts, 0)
    return {"x": synth.normal_bf16((int(off[-1]), K), 1.0, 1),
            "w": synth.student_t_outliers_bf16((experts, N, K), 4, 0.02, 5e-4, 20.0, 0),
            "m_offsets": off}


def _kd_sample_inputs(T=64):
    """CPU inputs for the oracle leg of the distillation workloads: the first
    positions of the same recipe (Qwen3-sized vocabulary)."""
    from learnable_scale_fake_gb300 import synth

    s, t, lab = synth.kd_logits(T, synth.KD_VOCAB, 0)
    return {"student": s, "teacher": t, "labels": lab}


def metric_name(workload, flops_kind):
    if flops_kind:
        return "fused NVFP4 fake-quant + grouped GEMM TFLOP/s"
    if workload.startswith("kd_"):
        return "distillation loss + student-logit gradient algorithmic HBM GB/s"
    return "fake-quant fwd+scale-grad algorithmic HBM GB/s"


def reference_arm(args):
    """--impl reference: the oracle, as it stands, on the host cores.  Inputs come
    from the seeded generators directly; nothing of the CUDA library runs."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    from learnable_scale_fake_gb300 import synth, workloads

    gen = {"grouped_nvfp4": lambda: synth.cfg3("cpu", 0, experts=8), "nvfp4_wa": lambda: synth.cfg2("cpu"),
           "grouped_nvfp4_fused": lambda: synth.cfg3("cpu", 0, experts=8),
           "nvfp4_wa_fused": lambda: synth.cfg2("cpu"), "int8_channel_fused": lambda: synth.cfg1("cpu"),
           "int4_fp8": lambda: synth.cfg4("cpu"), "int8_channel": lambda: synth.cfg1("cpu"),
           "observer_fp8": lambda: {"act": synth.head_normal_bf16(4096, 32, 128, 0.1, 10.0, 0)},
           "head_fp8_learned": lambda: {"act": synth.head_normal_bf16(4096, 32, 128, 0.1, 10.0, 0),
                                        "dy": synth.normal_bf16((4096, 32, 128), 1.0, 1)},
           "grouped_nvfp4_gemm": _gemm_sample_inputs,
           "kd_cakld": _kd_sample_inputs, "kd_topk": _kd_sample_inputs}
    inputs = gen[args.workload]()
    # the whole run (warm-up + timed steps) takes about a minute of oracle time
    per_step = 60.0 / max(1, args.steps + args.warmup)
    k, _, desc = oracle_pick(args.workload, inputs, target_s=per_step)
    runs = []
    for i in range(args.warmup + args.steps):
        r = oracle_run(args.workload, inputs, k)
        if i >= args.warmup:
            runs.append(r)
    tb = sum(r[0] for r in runs)
    ts = sum(r[2] for r in runs)
    gemm = args.workload == "grouped_nvfp4_gemm"
    unit = "TFLOP/s" if gemm else "GB/s"
    value = tb / ts / (1e12 if gemm else 1e9)
    threads = oracle.num_threads()
    line = {
        "impl": "reference",
        "metric": metric_name(args.workload, gemm),
        "value": round(value, 6), "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * ts / len(runs), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(workloads.CONFIGS[args.workload], sample=desc),
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------

def max_over_ranks(value, dist, device):
    import torch

    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse()
    plan = rank_plan(args.gpus, os.environ)
    if plan.startswith("error"):
        print(f"bench.py: {plan}", file=sys.stderr)
        sys.exit(2)
    if plan == "spawn":
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    if args.impl == "reference":
        reference_arm(args)
        return
    import torch

    from learnable_scale_fake_gb300 import _build, aqfq, workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist

        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    aqfq.lib()

    if args.experts is not None and args.workload in ("grouped_nvfp4", "grouped_nvfp4_fused",
                                                      "grouped_nvfp4_gemm"):
        wl = workloads.BUILDERS[args.workload](device, experts=args.experts)
    elif args.tokens is not None and args.workload in ("kd_cakld", "kd_topk"):
        wl = workloads.BUILDERS[args.workload](device, tokens=args.tokens)
    else:
        wl = workloads.BUILDERS[args.workload](device)
    stream = torch.cuda.Stream(device)
    small = wl.bytes_per_step < 1.5 * 129e6
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device) if small else None
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            wl.step(stream)
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps with no per-op events (a timing event
    # between two short kernels costs ~1-2 us of device time), then K more
    # steps with events around every op on the stream it is launched on, for
    # the per-op times and the roofline ----
    nops = len(wl.ops)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nops)] for _ in range(args.steps)]
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for k in range(args.steps):
            if flush is not None:  # the flush stays outside the step's events
                flush.fill_(k & 0xFF)
                sev[k][0].record(stream)
                wl.step(stream)
                sev[k][1].record(stream)
            else:
                wl.step(stream)
        t1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    with torch.cuda.stream(stream):
        i0.record(stream)
        for k in range(args.steps):
            if flush is not None:
                flush.fill_(k & 0xFF)
            wl.step(stream, hook=lambda i, st, end, k=k: ev[k][i][int(end)].record(st))
        i1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    if dist is not None:
        dist.barrier()
    per_op = [[ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
              for i in range(nops)]
    op_ms = [sum(v) / len(v) for v in per_op]
    if flush is None:
        step_ms = t0.elapsed_time(t1) / args.steps
        instr_ms = i0.elapsed_time(i1) / args.steps
    else:
        step_ms = sum(a.elapsed_time(b) for a, b in sev) / args.steps
        instr_ms = sum(op_ms) if not wl.phases else None
    step_ms = max_over_ranks(step_ms, dist, device)

    bytes_step = wl.bytes_per_step  # FLOPs per step for a contraction workload
    flops_kind = getattr(wl, "flops", None) is not None
    scale_unit = 1e12 if flops_kind else 1e9
    value = world * bytes_step / (step_ms * 1e-3) / scale_unit
    gelem = world * wl.elems_per_step / (step_ms * 1e-3) / 1e9
    if flops_kind:
        peak, peak_kind = tensor_peak()
    else:
        peak, peak_kind = hbm_peak()

    dom = max(range(nops), key=lambda i: op_ms[i])
    dom_op = wl.ops[dom]
    achieved = dom_op.bytes / (op_ms[dom] * 1e-3) / scale_unit
    roof = {"bound": "tensor" if flops_kind else "hbm", "kernel": dom_op.kernel, "op": dom_op.name,
            "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s" if flops_kind else "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": (f"{peak_kind} (MEASURED_PEAKS {'bf16_tflops' if flops_kind else 'hbm_gbs'})"
                            if peak_kind == "measured" else "fallback"),
            "traffic": stored_traffic(dom_op.name),
            "algorithmic_bytes_per_launch" if not flops_kind else "flops_per_launch": dom_op.bytes}
    # the same computation done the unfused way (reference path, for comparison)
    unfused = None
    for rop in getattr(wl, "reference_ops", []):
        with torch.cuda.stream(stream):
            for _ in range(2):
                rop.run(stream)
            torch.cuda.synchronize()
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            r0.record(stream)
            for _ in range(5):
                rop.run(stream)
            r1.record(stream)
        torch.cuda.synchronize()
        rms = r0.elapsed_time(r1) / 5
        unfused = {"op": rop.name, "ms": round(rms, 4),
                   "value": round(rop.bytes / (rms * 1e-3) / scale_unit, 1)}

    # ---- the same step launched as one CUDA graph (beside the eager timed
    # region: timing events cannot sit inside a captured graph, so per-op times
    # and the roofline come from the eager region above) ----
    graph = None
    if not args.no_graph:
        # every rank reaches the same collectives whether or not its capture
        # works; a failure anywhere shows as +inf in the max over ranks
        g, why = None, None
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                wl.step(stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
            torch.cuda.synchronize()
        except Exception as ex:  # a step that cannot be captured: report why
            g, why = None, f"{type(ex).__name__}: {ex}"[:200]
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        gms = float("inf")
        if g is not None:
            gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            with torch.cuda.stream(stream):
                for k in range(args.steps):
                    if flush is not None:
                        flush.fill_(k & 0xFF)
                    gev[k][0].record(stream)
                    g.replay()
                    gev[k][1].record(stream)
            torch.cuda.synchronize()
            gms = sum(a.elapsed_time(b) for a, b in gev) / args.steps
            del g
        gms = max_over_ranks(gms, dist, device)
        if gms != float("inf"):
            graph = {"ms_per_step": round(gms, 4),
                     "value": round(world * bytes_step / (gms * 1e-3) / scale_unit, 1),
                     "steps": args.steps, "timing": "CUDA events around each replay"}
        else:
            graph = {"unavailable": why or "capture failed on another rank"}

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        host_in, host_out = wl.host_buffers()
        bi = sum(v.numel() * v.element_size() for v in host_in.values())
        bo = sum(v.numel() * v.element_size() for v in host_out.values())
        streams = (torch.cuda.Stream(device), stream, torch.cuda.Stream(device))
        n_e2e = max(3, min(args.steps, 20))
        wl.e2e_step(host_in, host_out, streams)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            wl.e2e_step(host_in, host_out, streams)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dist, device)
        e2e = {"value": round(world * bytes_step / (e2e_ms * 1e-3) / scale_unit, 2),
               "unit": "TFLOP/s" if flops_kind else "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_ms, 3),
               "steps": n_e2e, "pipelined_slices": len(getattr(wl, "slices", None) or [])}

    # ---- CPU oracle on a bounded sample (rank 0, one GPU) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle

        k, _, desc = oracle_pick(args.workload, wl.inputs, target_s=20.0)
        nbytes, elems, secs = oracle_run(args.workload, wl.inputs, k)
        threads = oracle.num_threads()
        cpu = {"value": round(nbytes / secs / scale_unit, 6), "unit": "TFLOP/s" if flops_kind else "GB/s",
               "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": round(secs, 2),
               "gelem_per_s": round(elems / secs / 1e9, 5)}
        # the same oracle on one thread, on a smaller sample
        oracle.set_num_threads(1)
        try:
            k1, _, desc1 = oracle_pick(args.workload, wl.inputs, target_s=6.0)
            nb1, _, s1 = oracle_run(args.workload, wl.inputs, k1)
        finally:
            oracle.set_num_threads(threads)
        cpu["single_thread"] = {"value": round(nb1 / s1 / scale_unit, 6), "sample": desc1,
                                "seconds": round(s1, 2)}

    if rank == 0:
        metric = metric_name(args.workload, flops_kind)
        line = {
            "metric": metric, "value": round(value, 1),
            "unit": "TFLOP/s" if flops_kind else "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "storage": "bf16", "data": "synthetic",
            "config": dict(wl.config, l2=("flushed between steps (256 MiB write)" if small
                                          else "inputs larger than L2"),
                           parallelism=f"replicas x{world}",
                           **({"concurrent_phases": [[[wl.ops[i].name for i in lane] for lane in ph]
                                                     for ph in wl.phases]} if wl.phases else {})),
            "gelem_per_s": round(gelem, 2),
            "pct_of_peak": round(100 * value / world / peak, 1),
            "pct_hbm_nominal_8tbs": (None if flops_kind else
                                     round(100 * value / world / NOMINAL_HBM_GBS, 1)),
            "per_op_ms": {op.name: round(op_ms[i], 4) for i, op in enumerate(wl.ops)},
            "per_op_timing": ("CUDA events around each op on its own stream, in a second "
                              f"region of {args.steps} steps"
                              + (f"; that region's step {round(instr_ms, 4)} ms" if instr_ms else "")),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "unfused_path": unfused,
            "graph": graph,
            "gpu_launches": args.steps * sum(op.launches for op in wl.ops),
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
