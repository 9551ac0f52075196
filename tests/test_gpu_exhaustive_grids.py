"""Every binary32 value through the kernels' grid rounding, against the oracle.

The fake-quant kernels turn each quotient v = x / s into a code: E4M3 and
E2M1 by saturating round-to-nearest-even conversion of |v| with the sign of v
on the code, INT8 / INT4 by clamping and round-half-even (AngelSlim mcore_qad
article, section 3: formats fp8, nvfp4, w8a8, w4a16).  Here the GPU applies
that step (aqfq_selftest_grid_codes, the same device functions) to all 2^32
binary32 bit patterns but NaN, and each code is compared with the oracle's.

The oracle encodes by trying every grid value, far too slow for 2^32 calls,
so its answers are taken where they can change: the oracle maps |v| to codes
monotonically, so for every pair of neighbouring grid values the oracle is
asked at their midpoint and one binary32 step either side, which gives the
smallest |v| of each code; the expected code of any v is then the number of
such boundaries at or below |v| (a sorted search on the GPU), with the sign
bit of v.  The construction is itself checked against direct oracle calls on
random binary32 values and on infinities.
"""
import numpy as np
import pytest
import torch

import oracle
from learnable_scale_fake_gb300 import aqfq
from paritylib import dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
Q = aqfq.qspec


def _f32(x):
    return float(np.float32(x))


def _up(x):
    return _f32(np.nextafter(np.float32(x), np.float32(np.inf)))


def _down(x):
    return _f32(np.nextafter(np.float32(x), np.float32(-np.inf)))


def _fp_boundaries(decode, encode, maxcode):
    """Smallest |v| (binary32) of each magnitude code 1..maxcode, from oracle calls."""
    grid = [decode(c) for c in range(maxcode + 1)]
    assert all(a < b for a, b in zip(grid, grid[1:])), "codes ascend with their values"
    bounds = []
    for c in range(maxcode):
        m = (grid[c] + grid[c + 1]) / 2
        assert _f32(m) == m  # a binary32 value
        assert encode(_down(m)) == c and encode(_up(m)) == c + 1
        bounds.append(m if encode(m) == c + 1 else _up(m))
    return np.array(bounds, np.float32)


def _int_boundaries(qmin, qmax):
    """Smallest v (binary32) of each integer code qmin + 1 .. qmax, from oracle calls."""
    bounds = []
    for k in range(qmin, qmax):
        m = k + 0.5
        assert oracle.int_round(_down(m), qmin, qmax) == k
        assert oracle.int_round(_up(m), qmin, qmax) == k + 1
        bounds.append(m if oracle.int_round(m, qmin, qmax) == k + 1 else _up(m))
    return np.array(bounds, np.float32)


def _expected(kind, bounds, v, qmin=0, bits=8):
    """Expected codes of v (float32 tensor) from the boundaries (torch)."""
    if kind == "fp":
        mag = torch.searchsorted(bounds, v.abs(), right=True)
        sign = (v.view(torch.int32) < 0).to(torch.int64) << (bits - 1)
        return (mag | sign).to(torch.uint8)
    q = torch.searchsorted(bounds, v, right=True) + qmin
    return (q & ((1 << bits) - 1)).to(torch.uint8)


def _oracle_code(kind, v, qmin=0, qmax=0, bits=8):
    if kind == "e4m3":
        return oracle.e4m3_encode(v)
    if kind == "e2m1":
        return oracle.e2m1_encode(v)
    return int(oracle.int_round(v, qmin, qmax)) & ((1 << bits) - 1)


CASES = [
    # name, spec, kind for the oracle, boundaries, expected-code form, qmin, code bits
    ("e4m3", Q(aqfq.FP8_E4M3, aqfq.PER_TENSOR), "e4m3",
     lambda: _fp_boundaries(oracle.e4m3_decode, oracle.e4m3_encode, 0x7E), "fp", 0, 8),
    ("e2m1", Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16), "e2m1",
     lambda: _fp_boundaries(oracle.e2m1_decode, oracle.e2m1_encode, 7), "fp", 0, 4),
    ("int8", Q(aqfq.INT8, aqfq.PER_TENSOR, qmin=-128, qmax=127), "int",
     lambda: _int_boundaries(-128, 127), "int", -128, 8),
    ("int8_sym", Q(aqfq.INT8, aqfq.PER_TENSOR, qmin=-127, qmax=127), "int",
     lambda: _int_boundaries(-127, 127), "int", -127, 8),
    ("int4", Q(aqfq.INT4, aqfq.PER_TENSOR, qmin=-8, qmax=7), "int",
     lambda: _int_boundaries(-8, 7), "int", -8, 4),
]


@pytest.mark.parametrize("name,sp,okind,mkbounds,ekind,qmin,bits", CASES, ids=[c[0] for c in CASES])
def test_every_binary32_value(name, sp, okind, mkbounds, ekind, qmin, bits):
    d = dev()
    bounds = mkbounds()
    qmax = sp.qmax
    # the boundary construction against direct oracle calls: random binary32
    # values of every magnitude, signed zeros and infinities
    rng = np.random.default_rng(17)
    probe = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    probe = np.concatenate([probe[~np.isnan(probe)], np.float32([0.0, -0.0, np.inf, -np.inf])])
    want = np.array([_oracle_code(okind, float(x), qmin, qmax, bits) for x in probe], np.uint8)
    bt = torch.from_numpy(bounds).to(d)
    got = _expected(ekind, bt, torch.from_numpy(probe).to(d), qmin, bits).cpu().numpy()
    assert np.array_equal(got, want), "the boundary table disagrees with the oracle"
    # every binary32 bit pattern, 2^28 at a time
    chunk = 1 << 28
    codes = torch.empty(chunk, dtype=torch.uint8, device=d)
    checked = 0
    for c in range((1 << 32) // chunk):
        # the int32 values [-2^31, 2^31) are exactly the 2^32 bit patterns
        bitsv = (torch.arange(c * chunk, (c + 1) * chunk, dtype=torch.int64, device=d) - (1 << 31)).to(torch.int32)
        v = bitsv.view(torch.float32)
        aqfq.aqfq_selftest_grid_codes(sp, v, codes)
        keep = ~torch.isnan(v)
        exp = _expected(ekind, bt, v, qmin, bits)
        bad = (codes != exp) & keep
        nbad = int(bad.sum())
        if nbad:
            i = int(torch.nonzero(bad)[0])
            raise AssertionError(f"{nbad} codes differ in chunk {c}: v bits {int(bitsv[i]) & 0xFFFFFFFF:#010x} "
                                 f"gpu {int(codes[i]):#04x} oracle {int(exp[i]):#04x}")
        checked += int(keep.sum())
        del bitsv, v, keep, exp, bad
    assert checked == (1 << 32) - 2 * ((1 << 23) - 1)  # every pattern but the NaNs
