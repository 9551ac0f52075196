"""Seeded synthetic inputs for the fake-quant path.

This module only draws random tensors with the shapes and value distributions
of the workloads (weights, activations, upstream gradients, and free-standing
random scales for tests).  It holds none of the method's arithmetic: no
quantization, no scale initialisation, no gradient.  Both the CUDA path's
tests/benchmark and the CPU oracle are fed from here.

All draws go through an explicit ``torch.Generator`` seeded per tensor, so a
(seed, device) pair always gives the same tensor.  Values are drawn in fp32
and rounded to BF16 by torch's conversion.
"""
from __future__ import annotations

import math

import torch

# Workload shapes (MoE experts from a Qwen3-30B-A3B-sized layer: 128 experts,
# hidden 2048, expert intermediate 768, gate_up = 2 * 768 rows).
CFG1_W = (256, 512)
CFG2_W = (4096, 4096)
CFG2_A = (8192, 4096)
CFG3_GATE_UP = (128, 1536, 2048)
CFG3_DOWN = (128, 2048, 768)
CFG4_STACK = (128, 1536, 2048)
CFG4_DENSE = (8192, 8192)
CFG5_ACT = (65536, 32, 128)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _chunks(n0: int, per_row: int, budget: int = 1 << 26):
    """Split a leading dimension so one chunk holds about `budget` elements."""
    step = max(1, budget // max(1, per_row))
    for i in range(0, n0, step):
        yield i, min(n0, i + step)


def normal_bf16(shape, std, seed, device="cpu"):
    """x ~ N(0, std^2), rounded to BF16."""
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for a, b in _chunks(shape[0], flat.shape[1]):
        flat[a:b] = (torch.randn((b - a, flat.shape[1]), generator=g, device=device) * std).to(
            torch.bfloat16)
    return out


def normal_outliers_bf16(shape, std, p, mult, seed, device="cpu"):
    """x ~ N(0, std^2); each element independently (probability p) multiplied by mult."""
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for a, b in _chunks(shape[0], flat.shape[1]):
        z = torch.randn((b - a, flat.shape[1]), generator=g, device=device) * std
        m = torch.rand((b - a, flat.shape[1]), generator=g, device=device) < p
        z = torch.where(m, z * mult, z)
        flat[a:b] = z.to(torch.bfloat16)
    return out


def student_t_outliers_bf16(shape, nu, scale, p, mult, seed, device="cpu"):
    """x = scale * t_nu (t = Z / sqrt(chi2_nu / nu), nu integer), with iid
    Bernoulli(p) positions multiplied by mult."""
    nu = int(nu)
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for a, b in _chunks(shape[0], flat.shape[1], budget=1 << 25):
        n = (b - a, flat.shape[1])
        z = torch.randn(n, generator=g, device=device)
        chi2 = torch.zeros(n, device=device)
        for _ in range(nu):
            chi2.add_(torch.randn(n, generator=g, device=device).square_())
        t = z / torch.sqrt(chi2 / nu)
        m = torch.rand(n, generator=g, device=device) < p
        t = torch.where(m, t * mult, t) * scale
        flat[a:b] = t.to(torch.bfloat16)
    return out


def head_normal_bf16(T, H, D, lo, hi, seed, device="cpu"):
    """x[t, h, d] ~ N(0, sigma_h^2) with sigma_h log-uniform in [lo, hi]."""
    g = _gen(seed, device)
    u = torch.rand(H, generator=g, device=device)
    sigma = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=device)
    for a, b in _chunks(T, H * D):
        z = torch.randn((b - a, H, D), generator=g, device=device) * sigma.view(1, H, 1)
        out[a:b] = z.to(torch.bfloat16)
    return out


def loguniform_f32(shape, lo, hi, seed, device="cpu"):
    """Free-standing random positive fp32 values, log-uniform in [lo, hi]
    (used as stand-ins for learned scales after training has moved them)."""
    g = _gen(seed, device)
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float64)
    return torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).to(torch.float32)


def bf16_bits(t: torch.Tensor):
    """BF16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def from_bits(a, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> BF16 tensor."""
    import numpy as np

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


# ---- the five workloads (recipes; seeds fixed per tensor) -----------------------

def cfg1(device="cpu", seed=0):
    """INT8 per-channel weight [256,512] ~ N(0, 0.02^2); upstream grad ~ N(0,1)."""
    return {"w": normal_bf16(CFG1_W, 0.02, seed, device),
            "dy": normal_bf16(CFG1_W, 1.0, seed + 1, device)}


def cfg2(device="cpu", seed=0):
    """NVFP4 weight [4096,4096] ~ N(0, 0.02^2); activations [8192,4096] ~ N(0,1)
    with 0.1 % element outliers x30; upstream grads ~ N(0,1)."""
    return {"w": normal_bf16(CFG2_W, 0.02, seed, device),
            "dy_w": normal_bf16(CFG2_W, 1.0, seed + 1, device),
            "a": normal_outliers_bf16(CFG2_A, 1.0, 1e-3, 30.0, seed + 2, device),
            "dy_a": normal_bf16(CFG2_A, 1.0, seed + 3, device)}


def cfg3(device="cpu", seed=0, experts=None):
    """Grouped MoE expert stacks, Student-t(4) * 0.02 with 0.05 % outliers x20;
    upstream grads ~ N(0,1).  `experts` truncates the expert axis (sampling)."""
    gu = CFG3_GATE_UP if experts is None else (experts,) + CFG3_GATE_UP[1:]
    dn = CFG3_DOWN if experts is None else (experts,) + CFG3_DOWN[1:]
    return {"gate_up": student_t_outliers_bf16(gu, 4, 0.02, 5e-4, 20.0, seed, device),
            "down": student_t_outliers_bf16(dn, 4, 0.02, 5e-4, 20.0, seed + 1, device),
            "dy_gate_up": normal_bf16(gu, 1.0, seed + 2, device),
            "dy_down": normal_bf16(dn, 1.0, seed + 3, device)}


def cfg4(device="cpu", seed=0):
    """INT4 g128 stack [128,1536,2048] and FP8 dense [8192,8192], both N(0, 0.02^2);
    upstream grads ~ N(0,1)."""
    return {"stack": normal_bf16(CFG4_STACK, 0.02, seed, device),
            "dy_stack": normal_bf16(CFG4_STACK, 1.0, seed + 1, device),
            "dense": normal_bf16(CFG4_DENSE, 0.02, seed + 2, device),
            "dy_dense": normal_bf16(CFG4_DENSE, 1.0, seed + 3, device)}


def cfg5(device="cpu", seed=0):
    """Activations [65536 tokens, 32 heads, 128] with per-head std log-uniform in [0.1, 10]."""
    T, H, D = CFG5_ACT
    return {"act": head_normal_bf16(T, H, D, 0.1, 10.0, seed, device)}


def routing_counts(E, total, seed, skew=0.3, device="cpu"):
    """Tokens per expert for `total` routed rows: multinomial with expert
    popularity exp(N(0, skew^2)) (a mildly unbalanced router).  int64 [E]."""
    g = _gen(seed, "cpu")
    pop = torch.exp(torch.randn(E, generator=g, dtype=torch.float64) * skew)
    idx = torch.multinomial(pop / pop.sum(), total, replacement=True, generator=g)
    return torch.bincount(idx, minlength=E).to(device)


# ---- distillation logits ------------------------------------------------------------

# Qwen3-sized vocabulary; 4096 positions per step
KD_VOCAB = 151936
KD_TOKENS = 4096


def kd_logits(T, V, seed, device="cpu", sigma=2.0, noise=0.3, ignore=0.1, hit=0.7):
    """Teacher logits ~ N(0, sigma^2) with, at each position, one favoured
    token raised by U(4, 12); student logits = teacher + N(0, noise^2) (the
    same frozen model seen through fake-quantized weights); labels: the
    favoured token with probability `hit`, else uniform over the vocabulary,
    and -100 (no loss) at a fraction `ignore` of positions.
    Returns (student [T, V] BF16, teacher [T, V] BF16, labels int32 [T])."""
    g = _gen(seed, device)
    teacher = torch.empty((T, V), dtype=torch.bfloat16, device=device)
    student = torch.empty_like(teacher)
    fav = torch.randint(0, V, (T,), generator=g, device=device)
    lift = 4.0 + 8.0 * torch.rand(T, generator=g, device=device)
    for a, b in _chunks(T, V):
        t = torch.randn((b - a, V), generator=g, device=device) * sigma
        t[torch.arange(b - a, device=device), fav[a:b]] += lift[a:b]
        teacher[a:b] = t.to(torch.bfloat16)
        student[a:b] = (teacher[a:b].float() +
                        torch.randn((b - a, V), generator=g, device=device) * noise).to(torch.bfloat16)
    pick = torch.rand(T, generator=g, device=device) < hit
    other = torch.randint(0, V, (T,), generator=g, device=device)
    labels = torch.where(pick, fav, other)
    labels = torch.where(torch.rand(T, generator=g, device=device) < ignore,
                         torch.full_like(labels, -100), labels)
    return student, teacher, labels.to(torch.int32)
