"""Fused NVFP4 weight fake-quant + grouped GEMM (tcgen05) against the oracle.

Exactness of the in-kernel fake-quant: with one-hot activation rows, every
output is a single weight element times 1 (exact in any summation order), so
y must equal the oracle's w_hat bit for bit.  General inputs: FP32
accumulation of K products (each exact: BF16 x BF16) then rounding to BF16:
|y - ref| <= 2^-8 |ref| + K 2^-24 sum_k |x w_hat| (a bound, not a fit)."""
import numpy as np
import pytest
import torch

import oracle
from learnable_scale_fake_gb300 import aqfq, synth
from paritylib import bits, dev

pytestmark = pytest.mark.gpu


def _inputs(E, N, K, sizes, seed, onehot=False):
    w = synth.student_t_outliers_bf16((E, N, K), 4, 0.02, 5e-3, 20.0, seed)
    s = synth.loguniform_f32((E * N * K // 16,), 2e-3, 2e-2, seed + 1)
    g = synth.loguniform_f32((E,), 2e-5, 1e-4, seed + 2)
    M = int(sum(sizes))
    if onehot:
        gen = torch.Generator().manual_seed(seed + 3)
        cols = torch.randint(0, K, (M,), generator=gen)
        x = torch.zeros((M, K), dtype=torch.bfloat16)
        x[torch.arange(M), cols] = 1.0
    else:
        x = synth.normal_bf16((max(M, 1), K), 1.0, seed + 3)[:M]
    off = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]), dtype=torch.int32)
    return x, off, w, s, g


def _run(x, off, w, s, g):
    d = dev()
    E, N, K = w.shape
    y = torch.full((x.shape[0], N), float("nan"), dtype=torch.bfloat16, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    aqfq.aqfq_grouped_qdq_gemm(x.to(d).contiguous(), off.to(d), w.to(d), s.to(d), g.to(d), y, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "a pipeline wait timed out"
    return y.cpu()


def test_gemm_single_tile_onehot_exact():
    x, off, w, s, g = _inputs(1, 128, 64, [128], 200, onehot=True)
    y = _run(x, off, w, s, g)
    ref, _ = oracle.grouped_qdq_gemm(bits(x), off.numpy(), bits(w), s.numpy(), g.numpy())
    assert np.array_equal(bits(y), bits(torch.from_numpy(ref).to(torch.bfloat16)))


@pytest.mark.parametrize("E,N,K,sizes", [(3, 256, 128, [128, 200, 57]), (4, 384, 512, [0, 300, 1, 130]),
                                         (2, 128, 128, [1100, 513]), (3, 128, 64, [512, 0, 1024])])
def test_gemm_onehot_exact_ragged(E, N, K, sizes):
    x, off, w, s, g = _inputs(E, N, K, sizes, 210 + E, onehot=True)
    y = _run(x, off, w, s, g)
    ref, _ = oracle.grouped_qdq_gemm(bits(x), off.numpy(), bits(w), s.numpy(), g.numpy())
    yb, rb = bits(y), bits(torch.from_numpy(ref).to(torch.bfloat16))
    assert np.array_equal(yb, rb), f"{np.count_nonzero(yb != rb)} of {yb.size} differ"


@pytest.mark.parametrize("E,N,K,sizes", [(1, 128, 64, [77]), (5, 256, 1024, [256, 0, 129, 64, 383]),
                                         (2, 128, 2048, [300, 212])])
def test_gemm_random_within_bound(E, N, K, sizes):
    x, off, w, s, g = _inputs(E, N, K, sizes, 230 + E, onehot=False)
    y = _run(x, off, w, s, g).double().numpy()
    ref, absref = oracle.grouped_qdq_gemm(bits(x), off.numpy(), bits(w), s.numpy(), g.numpy())
    tol = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -24 * absref
    err = np.abs(y - ref)
    assert np.all(err <= tol), f"worst excess {(err - tol).max()} at {np.unravel_index(np.argmax(err - tol), err.shape)}"
    # typical error is far below the bound
    rel = err / np.maximum(np.abs(ref), 1e-30)
    assert np.median(rel) < 2.0 ** -8


def _e4m3_midpoints():
    """Midpoints between consecutive positive finite E4M3 values, and the
    saturation threshold halfway between 448 and the next step (480)."""
    vals = []
    for c in range(0x7F):  # 0x7F is NaN
        e, m = c >> 3, c & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    vals = np.array(sorted(set(vals)))
    return np.concatenate([(vals[1:] + vals[:-1]) / 2, [464.0]])


def test_gemm_block_scale_quotient_at_e4m3_midpoints():
    """Block scales whose quotient S_b / g lies within a few binary32 ulps of
    an E4M3 rounding midpoint (where a quotient off by one ulp changes the
    block's code), plus zero, subnormal, tiny and huge quotients that leave the
    kernel's short division path: one-hot rows make Y = w_hat^T bit for bit."""
    E, N, K = 2, 128, 1024
    rng = np.random.default_rng(77)
    g = (rng.uniform(1.0, 2.0, E) * 3e-5).astype(np.float32)
    mids = _e4m3_midpoints()
    deltas = np.array([0.0, 2.0 ** -24, -2.0 ** -24, 2.0 ** -23, -2.0 ** -23, 3 * 2.0 ** -24, -3 * 2.0 ** -24])
    nb = N * K // 16
    s = np.empty((E, nb), dtype=np.float32)
    for e in range(E):
        combo = rng.permutation(np.array([(m, d) for m in mids for d in deltas]))
        reps = np.resize(combo, (nb, 2))
        s[e] = (reps[:, 0] * float(g[e]) * (1.0 + reps[:, 1])).astype(np.float32)
        special = np.array([0.0, 1e-40, float(g[e]) * 2.0 ** -35, float(g[e]) * 2.0 ** -29,
                            float(g[e]) * 2.0 ** 101, float(g[e]) * 500.0, 1e30], dtype=np.float32)
        s[e, rng.choice(nb, special.size * 8, replace=False)] = np.tile(special, 8)
    w = synth.normal_bf16((E, N, K), 0.02, 78)
    M = E * K
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    x[torch.arange(M), torch.arange(M) % K] = 1.0
    off = torch.tensor([0, K, 2 * K], dtype=torch.int32)
    st, gt = torch.from_numpy(s.reshape(-1)), torch.from_numpy(g)
    y = _run(x, off, w, st, gt)
    ref, _ = oracle.grouped_qdq_gemm(bits(x), off.numpy(), bits(w), st.numpy(), gt.numpy())
    yb, rb = bits(y), bits(torch.from_numpy(ref).to(torch.bfloat16))
    assert np.array_equal(yb, rb), f"{np.count_nonzero(yb != rb)} of {yb.size} differ"


def test_gemm_many_experts_beyond_one_search_batch():
    """300 experts (the tile search takes experts 128 at a time), ragged sizes
    with empty experts and one past a 512-row group: one-hot rows exact."""
    rng = np.random.default_rng(41)
    sizes = rng.integers(0, 40, 300)
    sizes[::7] = 0
    sizes[250] = 530
    x, off, w, s, g = _inputs(300, 128, 64, sizes.tolist(), 250, onehot=True)
    y = _run(x, off, w, s, g)
    ref, _ = oracle.grouped_qdq_gemm(bits(x), off.numpy(), bits(w), s.numpy(), g.numpy())
    yb, rb = bits(y), bits(torch.from_numpy(ref).to(torch.bfloat16))
    assert np.array_equal(yb, rb), f"{np.count_nonzero(yb != rb)} of {yb.size} differ"


def test_gemm_offsets_clamped_to_rows():
    """Offsets below 0 or beyond total_m are clamped to [0, total_m]: the kernel
    computes the clamped experts and touches no row outside Y."""
    x, _, w, s, g = _inputs(2, 128, 128, [130, 70], 240, onehot=True)
    off = torch.tensor([-7, 130, 260], dtype=torch.int32)
    y = _run(x, off, w, s, g)
    ref, _ = oracle.grouped_qdq_gemm(bits(x), [0, 130, 200], bits(w), s.numpy(), g.numpy())
    assert np.array_equal(bits(y), bits(torch.from_numpy(ref).to(torch.bfloat16)))


def test_gemm_argument_checks():
    d = dev()
    x = torch.zeros((16, 64), dtype=torch.bfloat16, device=d)
    w = torch.zeros((1, 96, 64), dtype=torch.bfloat16, device=d)  # N % 128 != 0
    off = torch.tensor([0, 16], dtype=torch.int32, device=d)
    s = torch.ones(96 * 4, device=d)
    g = torch.ones(1, device=d)
    y = torch.empty((16, 96), dtype=torch.bfloat16, device=d)
    with pytest.raises(aqfq.AqfqError):
        aqfq.aqfq_grouped_qdq_gemm(x, off, w, s, g, y)


def test_bounded_wait_gives_up_and_context_survives():
    """A device wait that nothing completes gives up after its poll limit and
    raises the flag; the context stays usable (a GEMM right after is exact)."""
    d = dev()
    flag = torch.zeros(1, dtype=torch.int32, device=d)
    aqfq.aqfq_selftest_wait_timeout(flag, 1 << 12)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    x, off, w, s, g = _inputs(1, 128, 64, [128], 201, onehot=True)
    y = _run(x, off, w, s, g)
    ref, _ = oracle.grouped_qdq_gemm(bits(x), off.numpy(), bits(w), s.numpy(), g.numpy())
    assert np.array_equal(bits(y), bits(torch.from_numpy(ref).to(torch.bfloat16)))
