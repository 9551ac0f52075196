"""Element quotients placed on every rounding midpoint of every grid.

The forward and the gradient divide each element by its scale, v = fl32(x/s),
then round v to the format's grid (AngelSlim mcore_qad article, section 3:
formats nvfp4 / fp8 / w4a16 / w8a8; the gradient flows to the scale through
that rounding, section 2.3).  Where v sits on a rounding midpoint of the grid,
or a few units in the last place beside one, a quotient one ulp off flips the
code, the dequantised value and the gradient term.  The streaming kernels form
v with a per-chunk reciprocal and a correction step instead of a division per
element, so this is where they could part from the definition.

Each case below builds units whose quotient is exactly a chosen binary32
target: for every midpoint m of the grid (and the clamp boundary), the targets
m and its 1, 2, 3 ulp neighbours on both sides; for several BF16 magnitudes x
(random mantissas, plus a huge and a tiny x whose scales fall outside the
reciprocal path's range) the scale s is searched among binary32 values near
x/m so that fl32(x/s) equals the target (numpy's binary32 division is IEEE).
A unit holds +x and -x alternately, so negative midpoints are covered too.
Through the C ABI the GPU's codes, x_hat and STE input gradient must equal the
oracle's bit for bit and each scale gradient must lie within the tolerance;
every target must be reached by at least one unit.
"""
import numpy as np
import pytest
import torch

import oracle
from learnable_scale_fake_gb300 import aqfq
from paritylib import assert_grad_close, gpu_fwd, gpu_grad, oracle_fwd, oracle_grad

pytestmark = pytest.mark.gpu
Q = aqfq.qspec


def _bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _magnitudes():
    rng = np.random.default_rng(3)
    small = np.exp(rng.uniform(np.log(2.0 ** -8), np.log(2.0 ** -4), 8))
    return _bf16(np.concatenate([small, [1.3 * 2.0 ** 90, 1.7 * 2.0 ** -100]])).astype(np.float32)


XS = _magnitudes()


def _e4m3_grid():
    vals = {abs(oracle.e4m3_decode(c)) for c in range(256)}
    return np.array(sorted(v for v in vals if np.isfinite(v)))


def _midpoints(kind, qmax=None):
    """Positive rounding midpoints of the grid, then its clamp boundary (and,
    for the integer grids, the magnitude of qmin)."""
    if kind == "int":
        return np.concatenate([np.arange(qmax + 1) + 0.5, [float(qmax), float(qmax + 1)]])
    if kind == "e4m3":
        g = _e4m3_grid()
        return np.concatenate([(g[:-1] + g[1:]) / 2, [448.0]])
    return np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])  # E2M1 grid 0 .. 6


def _targets(base):
    """(target id, binary32 target) for every base value and its +-1..3 ulp
    neighbours."""
    t0 = base.astype(np.float32)
    assert np.array_equal(t0.astype(np.float64), base)  # midpoints are binary32 values
    ids, ts = [], []
    for k in range(-3, 4):
        t = t0.copy()
        for _ in range(abs(k)):
            t = np.nextafter(t, np.float32(np.inf if k > 0 else 0.0))
        ids.append(np.arange(t0.size) * 7 + (k + 3))
        ts.append(t)
    return np.concatenate(ids), np.concatenate(ts)


def _search(param0, quotient, target, span=32):
    """The binary32 value p nearest param0 (walking outwards, at most `span`
    ulps each way) with quotient(p) == target, else NaN; all arrays."""
    best = np.full_like(param0, np.nan)
    up, dn = param0.copy(), param0.copy()
    for _ in range(span):
        for c in (up, dn):
            with np.errstate(all="ignore"):
                hit = (quotient(c) == target) & np.isnan(best)
            best[hit] = c[hit]
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(0.0))
    return best


def _units(base):
    """Every (target, x) pair with a scale s such that fl32(x / s) == target:
    returns (target ids, x, s) of the pairs found; asserts every target id is
    reached."""
    ids, t = _targets(base)
    X = np.repeat(XS[None, :], t.size, 0).ravel()
    T = np.repeat(t[:, None], XS.size, 1).ravel()
    I = np.repeat(ids[:, None], XS.size, 1).ravel()
    s0 = (X.astype(np.float64) / T.astype(np.float64)).astype(np.float32)
    s = _search(s0, lambda c: X / c, T)
    ok = ~np.isnan(s)
    assert np.unique(I[ok]).size == ids.size, "a target quotient is not reachable"
    # the oracle's own binary32 quotient lands on the targets (a sample)
    for j in np.random.default_rng(0).choice(np.nonzero(ok)[0], 64, replace=False):
        assert oracle.div32(float(X[j]), float(s[j])) == float(T[j])
    return I[ok], X[ok], s[ok]


def _rows(x, width, anchor=None):
    """[units, width] BF16 rows of +x, -x, +x, ...; element 0 = anchor if given."""
    sign = np.where(np.arange(width) % 2 == 0, 1.0, -1.0).astype(np.float32)
    r = x[:, None] * sign[None, :]
    if anchor is not None:
        r[:, 0] = anchor
    return torch.tensor(r).to(torch.bfloat16)


def _dy(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def _compare(sp, x, scale, ts, seed):
    """GPU forward and gradient against the oracle on the same inputs."""
    dy = _dy(x.shape, seed)
    yg, cg, bg = gpu_fwd(sp, x, scale, ts)
    yo, co, bo = oracle_fwd(sp, x, scale, ts)
    assert np.array_equal(cg, co), f"{np.count_nonzero(cg != co)} codes differ"
    assert np.array_equal(yg, yo.reshape(yg.shape)), f"{np.count_nonzero(yg != yo)} x_hat differ"
    if bg is not None:
        assert np.array_equal(bg, bo), "block codes differ"
    dsg, dtg, dxg = gpu_grad(sp, x, dy, scale, ts)
    orc = oracle_grad(sp, x, dy, scale, ts)
    assert np.array_equal(dxg, orc["dx"].reshape(dxg.shape)), "STE input gradient differs"
    if dtg is not None:
        assert_grad_close(dtg, orc["dtensor_scale"], orc["dtensor_scale_abs"], what="dtensor_scale")
    else:
        assert_grad_close(dsg, orc["dscale"], orc["dscale_abs"])


INT8 = Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-128, qmax=127)
CASES = [
    # name, spec, grid, layout ("channel": [1, U, K]; "tensor": [U, 1, K]; "head": [1, U, K]), K
    ("int8_channel", INT8, ("int", 127), "channel", 16),
    ("int8_tensor", Q(aqfq.INT8, aqfq.PER_TENSOR, qmin=-128, qmax=127), ("int", 127), "tensor", 16),
    ("int8_channel_row_kernel", INT8, ("int", 127), "channel", 48),
    ("int4_g16", Q(aqfq.INT4, aqfq.PER_GROUP, group=16, qmin=-8, qmax=7), ("int", 7), "channel", 16),
    ("int4_g128", Q(aqfq.INT4, aqfq.PER_GROUP, group=128, qmin=-8, qmax=7), ("int", 7), "channel", 128),
    # grids whose one-comparison clamp test is exact (centre -1/2, +1/2) and
    # grids where it is not and the two comparisons stay (qmax or -qmin a power
    # of two: the quotient one ulp inside it, e.g. 1 - 2^-24, is a target)
    ("int4_g16_m4_3", Q(aqfq.INT4, aqfq.PER_GROUP, group=16, qmin=-4, qmax=3), ("int", 3), "channel", 16),
    ("int4_g16_m3_4", Q(aqfq.INT4, aqfq.PER_GROUP, group=16, qmin=-3, qmax=4), ("int", 3), "channel", 16),
    ("int4_g16_m2_1", Q(aqfq.INT4, aqfq.PER_GROUP, group=16, qmin=-2, qmax=1), ("int", 1), "channel", 16),
    ("int4_g16_m1_2", Q(aqfq.INT4, aqfq.PER_GROUP, group=16, qmin=-1, qmax=2), ("int", 1), "channel", 16),
    ("int8_channel_m65_64", Q(aqfq.INT8, aqfq.PER_CHANNEL, qmin=-65, qmax=64), ("int", 64), "channel", 16),
    ("fp8_channel", Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL), ("e4m3",), "channel", 16),
    ("fp8_channel_row_kernel", Q(aqfq.FP8_E4M3, aqfq.PER_CHANNEL), ("e4m3",), "channel", 48),
    ("fp8_tensor", Q(aqfq.FP8_E4M3, aqfq.PER_TENSOR), ("e4m3",), "tensor", 16),
    ("fp8_head", Q(aqfq.FP8_E4M3, aqfq.PER_HEAD), ("e4m3",), "head", 16),
]


@pytest.mark.parametrize("name,sp,grid,layout,K", CASES, ids=[c[0] for c in CASES])
def test_learned_scale_quotients_at_midpoints(name, sp, grid, layout, K):
    base = _midpoints(*grid) if grid[0] == "int" else _midpoints(grid[0])
    _, x, s = _units(base)
    rows = _rows(x, K)
    xt = rows[None] if layout in ("channel", "head") else rows[:, None]
    _compare(sp, xt, torch.from_numpy(s), None, seed=11)


def test_nvfp4_learned_block_scale_quotients_at_e2m1_midpoints():
    """Learned block scales: S_hat = dec(e) * g with g a non-unit binary32 per
    tensor (one unit per batch entry) and e among normal E4M3 codes;
    g is searched so that fl32(x / S_hat) hits each target."""
    codes = np.array([0x18, 0x2B, 0x38, 0x3B, 0x4D, 0x66])
    d = np.array([oracle.e4m3_decode(int(c)) for c in codes], np.float32)
    ids, t = _targets(_midpoints("e2m1"))
    # every (target, x, block code) combination
    T = np.repeat(t, XS.size * d.size)
    I = np.repeat(ids, XS.size * d.size)
    X = np.tile(np.repeat(XS, d.size), t.size)
    D = np.tile(d, t.size * XS.size)
    g0 = (X.astype(np.float64) / (T.astype(np.float64) * D)).astype(np.float32)
    g = _search(g0, lambda c: X / (D * c), T)
    ok = ~np.isnan(g) & (g >= 2.0 ** -100) & (g <= 2.0 ** 100)
    assert np.unique(I[ok]).size == ids.size, "a target quotient is not reachable"
    X, D, g = X[ok], D[ok], g[ok]
    sb = D * g  # S_b / g rounds back to the chosen code
    xt = _rows(X, 16)[:, None]
    sp = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16)
    _, _, bo = oracle_fwd(sp, xt, torch.from_numpy(sb), torch.from_numpy(g))
    want = np.array([oracle.e4m3_encode(float(v)) for v in D])
    assert np.array_equal(bo.reshape(-1), want), "the block codes are not the chosen ones"
    _compare(sp, xt, torch.from_numpy(sb), torch.from_numpy(g), seed=12)


def test_nvfp4_dynamic_block_scale_quotients_at_e2m1_midpoints():
    """Dynamic block scales (activations): element 0 of each block is the
    block's largest magnitude A, chosen so that fl32(A/6)/g rounds to a chosen
    E4M3 code; the learned tensor scale g is searched so that the other
    elements' quotients fl32(x / S_hat) hit each target below 6."""
    codes = np.array([0x20, 0x38, 0x3B, 0x4D])
    d = np.array([oracle.e4m3_decode(int(c)) for c in codes], np.float32)
    base = _midpoints("e2m1")[:-1]  # targets below the clamp: x stays below the anchor
    ids, t = _targets(base)
    T = np.repeat(t, XS.size * d.size)
    I = np.repeat(ids, XS.size * d.size)
    X = np.tile(np.repeat(XS, d.size), t.size)
    D = np.tile(d, t.size * XS.size)
    g0 = (X.astype(np.float64) / (T.astype(np.float64) * D)).astype(np.float32)
    with np.errstate(all="ignore"):
        A = _bf16(np.float32(6.0) * D * g0).astype(np.float32)
    g = _search(g0, lambda c: X / (D * c), T)
    ok = ~np.isnan(g) & np.isfinite(A) & (A > 0) & (X < A) & (g >= 2.0 ** -100) & (g <= 2.0 ** 100)
    # keep the units whose block code is the chosen one (fl32(fl32(A / 6) / g))
    with np.errstate(all="ignore"):
        q = (A / np.float32(6.0)) / g
    code = np.array([oracle.e4m3_encode(float(v)) if k else -1 for v, k in zip(q, ok)])
    want = np.array([oracle.e4m3_encode(float(v)) for v in D])
    ok &= code == want
    assert np.unique(I[ok]).size == ids.size, "a target quotient is not reachable"
    xt = _rows(X[ok], 16, anchor=A[ok])[:, None]
    sp = Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16, mode=aqfq.SCALE_DYNAMIC_BLOCK)
    _compare(sp, xt, None, torch.from_numpy(g[ok]), seed=13)
