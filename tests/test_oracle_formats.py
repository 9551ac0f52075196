"""Pins for the oracle's format primitives, against things other than itself:
torch's own float8_e4m3fn and bfloat16 conversions (library routines), numpy's
IEEE binary32 division and rint, closed forms of the format definitions, and
hand-derived tie cases (tests/golden/e2m1_ties.txt)."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore")


def _e4m3_grid_positive():
    return np.array([oracle.e4m3_decode(c) for c in range(0x7F)])


def test_e4m3_grid_by_enumeration():
    vals = [oracle.e4m3_decode(c) for c in range(256)]
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    pos = np.array(vals[:0x7F])
    assert np.all(np.diff(pos) > 0), "codes 0..0x7E must increase with the value"
    nz = pos[pos > 0]
    assert len(nz) == 126
    assert nz.max() == 448.0
    assert nz.min() == 2.0 ** -9
    assert min(v for v in nz if v >= 2.0 ** -6) == 2.0 ** -6  # smallest normal
    # negative half mirrors the positive half
    for c in range(0x7F):
        assert vals[c | 0x80] == -vals[c] or (vals[c] == 0 and math.copysign(1, vals[c | 0x80]) < 0)


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(ours[~nan]))


def test_e2m1_grid_closed_form():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(8):
        assert oracle.e2m1_decode(c) == mags[c]
        neg = oracle.e2m1_decode(c | 8)
        assert neg == -mags[c] and math.copysign(1.0, neg) == -1.0


def _e4m3_test_values(rng):
    grid = _e4m3_grid_positive()
    mids = (grid[1:] + grid[:-1]) / 2  # all exact in binary32
    vals = [mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
            np.nextafter(mids.astype(np.float32), np.float32(0)), grid,
            rng.standard_normal(4000) * 10, rng.standard_normal(4000) * 1e-2,
            np.exp(rng.uniform(np.log(1e-5), np.log(500), 4000)),
            np.array([0.0, 447.9, 448.0, 460, 464.0, 465, 1e6, 2.0 ** -10, 2.0 ** -11,
                      3 * 2.0 ** -11])]
    v = np.concatenate(vals).astype(np.float32)
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch():
    rng = np.random.default_rng(0)
    v = _e4m3_test_values(rng)
    ref = torch.from_numpy(v).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    bad = np.nonzero(ref != ours)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {v[bad[:5]]}: {ref[bad[:5]]} vs {ours[bad[:5]]}"


def test_e4m3_ties_go_to_even_code():
    grid = _e4m3_grid_positive()
    for c in range(0x7E):
        mid = float(np.float32((grid[c] + grid[c + 1]) / 2))
        got = oracle.e4m3_encode(mid)
        assert got in (c, c + 1) and got % 2 == 0
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-9) == 0x80
    assert oracle.e4m3_encode(1e30) == 0x7E and oracle.e4m3_encode(-1e30) == 0xFE


def test_e2m1_ties_golden():
    rows, _ = read_golden("e2m1_ties.txt")
    for inp, code, val in rows:
        c = oracle.e2m1_encode(float(inp))
        assert c == int(code, 16), (inp, hex(c), code)
        d = oracle.e2m1_decode(c)
        assert d == float(val) and math.copysign(1, d) == math.copysign(1, float(val))


def test_e2m1_encode_is_a_nearest_grid_point():
    rng = np.random.default_rng(1)
    grid = np.array([oracle.e2m1_decode(c) for c in range(8)])
    v = np.concatenate([rng.uniform(-8, 8, 20000), rng.standard_normal(2000) * 1e-3]).astype(
        np.float32)
    for x in v:
        c = oracle.e2m1_encode(float(x))
        q = oracle.e2m1_decode(c)
        a = min(abs(float(x)), 6.0)
        d = np.abs(grid - a)
        assert abs(abs(q) - a) == d.min()
        assert (c & 8 != 0) == bool(np.signbit(x))


def test_int_round_half_even_and_clamp():
    cases = {0.5: 0.0, 1.5: 2.0, 2.5: 2.0, -0.5: -0.0, -1.5: -2.0, -2.5: -2.0, 126.5: 126.0,
             127.5: 127.0, -128.5: -128.0, 1e9: 127.0, -1e9: -128.0, 0.49999997: 0.0}
    for v, q in cases.items():
        got = oracle.int_round(v, -128, 127)
        assert got == q and math.copysign(1, got) == math.copysign(1, q), (v, got)
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(5000) * 60).astype(np.float32)
    ref = np.clip(np.rint(v.astype(np.float64)), -8, 7)
    ours = np.array([oracle.int_round(float(x), -8, 7) for x in v])
    assert np.array_equal(ref, ours)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    # exact ties (low half 0x8000), values next to ties, subnormals, near overflow
    hi = rng.integers(0, 2 ** 16, 2000, dtype=np.uint64).astype(np.uint32) << 16
    extra = np.concatenate([hi | 0x8000, hi | 0x7FFF, hi | 0x8001,
                            rng.integers(1, 2 ** 23, 2000).astype(np.uint32),
                            np.array([0x7F7F8000, 0x7F7FFFFF, 0x00008000, 0x00018000],
                                     dtype=np.uint32)])
    f = np.concatenate([bits, extra]).view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.bf16_round(x) for x in f], dtype=np.uint16)
    bad = np.nonzero(ref != ours)[0]
    assert bad.size == 0, f"{bad.size} mismatches: {f[bad[:4]]} {ref[bad[:4]]} {ours[bad[:4]]}"


def test_div32_matches_ieee_binary32():
    rng = np.random.default_rng(4)
    a = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-38]).astype(
        np.float32)
    b = np.concatenate([np.exp(rng.uniform(-20, 20, 20000)),
                        np.exp(rng.uniform(-2, 2, 2000))]).astype(np.float32)
    with np.errstate(all="ignore"):
        ref = a / b
    ours = np.array([oracle.div32(float(x), float(y)) for x, y in zip(a, b)], dtype=np.float32)
    assert np.array_equal(ref.view(np.uint32), ours.view(np.uint32))
