"""Pins for the oracle's fake-quant forward, scale gradient, observer and scale
initialisation.  Each test checks the oracle against something other than
itself: torch's fake-quant operators (library), hand-worked fixtures under
tests/golden/, closed forms, and invariants (idempotence, odd symmetry,
power-of-two scale equivariance, shard merges, granularity consistency)."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from learnable_scale_fake_gb300 import synth

O = oracle


def bits(t):
    return synth.bf16_bits(t)


def f32_of_bits(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_of(vals):
    return bits(torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16))


# --------------------------------------------------------------------------------------
# forward: library cross-checks
# --------------------------------------------------------------------------------------

def test_int8_per_channel_matches_torch_fake_quantize_pow2_scales():
    """torch.fake_quantize_per_channel_affine multiplies by 1/scale; with
    power-of-two scales that equals the division, so the two must agree bit
    for bit (after the cast back to BF16)."""
    w = synth.normal_bf16((64, 256), 0.02, seed=11)
    g = torch.Generator().manual_seed(5)
    s = (2.0 ** torch.randint(-13, -6, (64,), generator=g)).to(torch.float32)
    ref = torch.fake_quantize_per_channel_affine(w.float(), s, torch.zeros(64, dtype=torch.int32),
                                                 0, -128, 127).to(torch.bfloat16)
    y, codes, _ = O.qdq_fwd(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127),
                            bits(w)[None], s.numpy(), want_codes=True)
    assert np.array_equal(y[0], bits(ref))
    # codes are the integers q with x_hat = q * s
    q = codes.view(np.int8)[0].astype(np.float64)
    assert np.array_equal((q * s.numpy()[:, None].astype(np.float64)).astype(np.float32),
                          ref.float().numpy())


def test_int8_per_channel_agrees_with_torch_on_random_scales():
    """With arbitrary scales torch's reciprocal-multiply may round v differently
    at exact ties only; everything else must agree."""
    w = synth.normal_bf16((128, 512), 0.02, seed=12)
    s = synth.loguniform_f32((128,), 1e-4, 4e-4, seed=13)
    ref = torch.fake_quantize_per_channel_affine(w.float(), s, torch.zeros(128, dtype=torch.int32),
                                                 0, -128, 127).to(torch.bfloat16)
    y, _, _ = O.qdq_fwd(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), bits(w)[None], s.numpy())
    mism = np.count_nonzero(y[0] != bits(ref))
    assert mism <= 5, mism


def test_fp8_per_channel_matches_torch_float8_cast():
    """E4M3 QDQ with power-of-two scales against torch's float8_e4m3fn cast."""
    w = synth.normal_bf16((64, 256), 0.02, seed=14)
    g = torch.Generator().manual_seed(6)
    s = (2.0 ** torch.randint(-16, -9, (64,), generator=g)).to(torch.float32)
    v = w.float() / s[:, None]
    ref = (v.clamp(-448, 448).to(torch.float8_e4m3fn).float() * s[:, None]).to(torch.bfloat16)
    y, codes, _ = O.qdq_fwd(O.spec(O.FP8_E4M3, O.PER_CHANNEL), bits(w)[None], s.numpy(),
                            want_codes=True)
    assert np.array_equal(y[0], bits(ref))
    ref_codes = v.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[0], ref_codes)


# --------------------------------------------------------------------------------------
# forward: hand-worked fixtures
# --------------------------------------------------------------------------------------

def test_nvfp4_block_golden():
    rows, kv = read_golden("nvfp4_block.txt")
    x = np.array([float(r[0]) for r in rows], np.float32)
    xb = bf16_bits_of(x)
    assert np.array_equal(f32_of_bits(xb), x), "fixture inputs must be exact in BF16"
    g = np.array([float(kv["g"][0])], np.float32)
    sb = np.array([float(kv["s_b"][0])], np.float32)
    sp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    y, codes, blk = O.qdq_fwd(sp, xb.reshape(1, 1, 16), sb, g, want_codes=True)
    assert blk[0, 0, 0] == int(kv["block_code"][0], 16)
    want_y = np.array([float(r[3]) for r in rows], np.float32)
    assert np.array_equal(y.reshape(-1), bf16_bits_of(want_y))
    assert [int(c) for c in codes.reshape(-1)] == [int(c, 16) for c in kv["codes"]]
    dy = bf16_bits_of(np.arange(1, 17, dtype=np.float32))
    gr = O.scale_grad(sp, xb.reshape(1, 1, 16), dy.reshape(1, 1, 16), sb, g)
    assert gr["dscale"][0] == float(kv["dscale"][0])
    terms = np.array([float(r[4]) for r in rows])
    assert gr["dscale_abs"][0] == np.sum(np.abs(terms * np.arange(1, 17)))
    # STE input gradient: dy where |v| < 6, zero where clamped
    clipped = np.abs(np.array([float(r[1]) for r in rows])) >= 6
    dx = f32_of_bits(gr["dx"].reshape(-1))
    assert np.array_equal(dx, np.where(clipped, 0, np.arange(1, 17)).astype(np.float32))


def test_int4_block_golden():
    rows, kv = read_golden("int4_block.txt")
    x = np.array([float(r[0]) for r in rows], np.float32)
    xb = bf16_bits_of(x).reshape(1, 1, 16)
    sp = O.spec(O.INT4, O.PER_GROUP, group=16, qmin=-8, qmax=7)
    s = np.ones(1, np.float32)
    y, codes, _ = O.qdq_fwd(sp, xb, s, want_codes=True)
    want = np.array([float(r[1]) for r in rows], np.float32)
    assert np.array_equal(y.reshape(-1), bf16_bits_of(want))  # includes the sign of -0
    assert [int(c) for c in codes.reshape(-1)] == [int(c, 16) for c in kv["codes"]]
    dy = bf16_bits_of(np.ones(16, np.float32)).reshape(1, 1, 16)
    gr = O.scale_grad(sp, xb, dy, s)
    assert gr["dscale"][0] == float(kv["dscale"][0])
    terms = np.array([float(r[3]) for r in rows])
    assert gr["dscale_abs"][0] == np.abs(terms).sum()


def test_fp8_init_scale_page_example():
    _, kv = read_golden("fp8_init_scale.txt")
    amax, want = float(kv["amax"][0]), float(kv["scale"][0])
    w = synth.normal_bf16((8, 32), 0.02, seed=15)
    wb = bits(w)
    wb[3, 7] = bf16_bits_of([-amax])[0]
    s, _ = O.scale_init(O.spec(O.FP8_E4M3, O.PER_TENSOR), wb[None])
    assert s[0] == np.float32(want)


# --------------------------------------------------------------------------------------
# forward: invariants
# --------------------------------------------------------------------------------------

LEARNED_SPECS = [
    ("int8_channel", O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), 4e-5, 4e-4),
    ("int8_sym_tensor", O.spec(O.INT8, O.PER_TENSOR, qmin=-127, qmax=127), 1e-4, 4e-4),
    ("int4_g128", O.spec(O.INT4, O.PER_GROUP, group=128, qmin=-8, qmax=7), 2e-3, 2e-2),
    ("int4_g16", O.spec(O.INT4, O.PER_GROUP, group=16, qmin=-8, qmax=7), 2e-3, 2e-2),
    ("fp8_channel", O.spec(O.FP8_E4M3, O.PER_CHANNEL), 2e-5, 2e-4),
    ("fp8_group32", O.spec(O.FP8_E4M3, O.PER_GROUP, group=32), 2e-5, 2e-4),
    ("fp8_head", O.spec(O.FP8_E4M3, O.PER_HEAD), 2e-5, 2e-4),
]


def _scale_count(sp, B, R, K):
    return {O.PER_TENSOR: B, O.PER_CHANNEL: B * R, O.PER_HEAD: R}.get(
        sp.gran, B * R * (K // max(sp.group, 1)))


@pytest.mark.parametrize("name,sp,lo,hi", LEARNED_SPECS, ids=[s[0] for s in LEARNED_SPECS])
def test_qdq_idempotent_learned(name, sp, lo, hi):
    B, R, K = 2, 24, 256
    x = bits(synth.normal_bf16((B, R, K), 0.02, seed=21))
    s = synth.loguniform_f32((_scale_count(sp, B, R, K),), lo, hi, seed=22).numpy()
    y1, c1, _ = O.qdq_fwd(sp, x, s, want_codes=True)
    y2, c2, _ = O.qdq_fwd(sp, y1, s, want_codes=True)
    assert np.array_equal(y1, y2)
    assert np.array_equal(c1, c2)


def test_nvfp4_learned_idempotent_and_odd():
    B, R, K = 3, 16, 128
    x = bits(synth.student_t_outliers_bf16((B, R, K), 4, 0.02, 5e-3, 20.0, seed=23))
    sp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    sb = synth.loguniform_f32((B * R * K // 16,), 2e-3, 2e-2, seed=24).numpy()
    g = synth.loguniform_f32((B,), 2e-5, 1e-4, seed=25).numpy()
    y1, c1, b1 = O.qdq_fwd(sp, x, sb, g, want_codes=True)
    y2, c2, b2 = O.qdq_fwd(sp, y1, sb, g, want_codes=True)
    assert np.array_equal(y1, y2) and np.array_equal(c1, c2) and np.array_equal(b1, b2)
    yn, _, _ = O.qdq_fwd(sp, x ^ np.uint16(0x8000), sb, g)
    assert np.array_equal(yn, y1 ^ np.uint16(0x8000))


def test_nvfp4_dynamic_odd_symmetry():
    x = bits(synth.normal_outliers_bf16((2, 32, 64), 1.0, 1e-2, 30.0, seed=26))
    sp = O.spec(O.NVFP4, O.PER_GROUP, group=16, mode=O.SCALE_DYNAMIC_BLOCK)
    g = np.array([0.01, 0.003], np.float32)
    y, _, blk = O.qdq_fwd(sp, x, None, g, want_codes=True)
    yn, _, blkn = O.qdq_fwd(sp, x ^ np.uint16(0x8000), None, g, want_codes=True)
    assert np.array_equal(yn, y ^ np.uint16(0x8000)) and np.array_equal(blk, blkn)


@pytest.mark.parametrize("fmt", [O.INT4, O.FP8_E4M3])
def test_symmetric_grid_odd_symmetry(fmt):
    sp = O.spec(fmt, O.PER_CHANNEL, qmin=-7, qmax=7)
    x = bits(synth.normal_bf16((1, 32, 128), 0.02, seed=27))
    s = synth.loguniform_f32((32,), 1e-3, 1e-2, seed=28).numpy()
    if fmt == O.FP8_E4M3:
        s = s / 100
    y, _, _ = O.qdq_fwd(sp, x, s)
    yn, _, _ = O.qdq_fwd(sp, x ^ np.uint16(0x8000), s)
    if fmt == O.FP8_E4M3:
        assert np.array_equal(yn, y ^ np.uint16(0x8000))
    else:  # integer code 0 dequantises to +0 on both sides
        assert np.array_equal(f32_of_bits(yn), -f32_of_bits(y))


@pytest.mark.parametrize("name,sp,lo,hi", LEARNED_SPECS[:5], ids=[s[0] for s in LEARNED_SPECS[:5]])
def test_pow2_scale_equivariance(name, sp, lo, hi):
    """QDQ(c*x; c*s) == c * QDQ(x; s) for c a power of two (no over/underflow)."""
    B, R, K = 1, 16, 256
    xt = synth.normal_bf16((B, R, K), 0.02, seed=29)
    s = synth.loguniform_f32((_scale_count(sp, B, R, K),), lo, hi, seed=30).numpy()
    y, c, _ = O.qdq_fwd(sp, bits(xt), s, want_codes=True)
    y8, c8, _ = O.qdq_fwd(sp, bits(xt * 8), (s * 8).astype(np.float32), want_codes=True)
    assert np.array_equal(y8, bits(synth.from_bits(y) * 8)) and np.array_equal(c, c8)


@pytest.mark.filterwarnings("ignore:All-NaN")
def test_int_codes_minimise_distance_bruteforce():
    """Every INT8 code is an argmin of |v - q| over the whole grid (ties to even),
    with v the correctly rounded binary32 quotient."""
    x = bits(synth.normal_bf16((1, 8, 512), 0.02, seed=31))
    s = synth.loguniform_f32((8,), 5e-5, 3e-4, seed=32).numpy()
    _, codes, _ = O.qdq_fwd(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), x, s,
                            want_codes=True)
    xf = f32_of_bits(x[0])
    v = (xf / s[:, None]).astype(np.float32).astype(np.float64)  # numpy binary32 division
    grid = np.arange(-128, 128, dtype=np.float64)
    d = np.abs(v[..., None] - grid)
    best = d.min(-1, keepdims=True)
    cand = np.where(d == best, grid, np.nan)
    even = np.where(np.isnan(cand), np.nan, np.where(cand % 2 == 0, cand, np.nan))
    pick = np.where(np.isnan(even).all(-1), np.nanmax(cand, -1), np.nanmax(even, -1))
    assert np.array_equal(codes[0].view(np.int8).astype(np.float64), pick)


def test_scale_indexing_by_slicing():
    """Each granularity equals per-tensor QDQ applied slice by slice (numpy
    slicing picks the unit; the scale comes from the unit's own index)."""
    B, R, K = 2, 3, 64
    x = bits(synth.normal_bf16((B, R, K), 0.02, seed=33))
    tn = O.spec(O.FP8_E4M3, O.PER_TENSOR)
    cases = [(O.spec(O.FP8_E4M3, O.PER_CHANNEL), B * R, lambda b, r, j: b * R + r, K),
             (O.spec(O.FP8_E4M3, O.PER_GROUP, group=32), B * R * 2, lambda b, r, j: (b * R + r) * 2 + j, 32),
             (O.spec(O.FP8_E4M3, O.PER_HEAD), R, lambda b, r, j: r, K)]
    for sp, n, idx, width in cases:
        s = synth.loguniform_f32((n,), 2e-5, 2e-4, seed=34).numpy()
        y, _, _ = O.qdq_fwd(sp, x, s)
        for b in range(B):
            for r in range(R):
                for j in range(K // width):
                    sl = slice(j * width, (j + 1) * width)
                    ys, _, _ = O.qdq_fwd(tn, x[b:b + 1, r:r + 1, sl], s[idx(b, r, j):idx(b, r, j) + 1])
                    assert np.array_equal(ys[0, 0], y[b, r, sl])
    # NVFP4: every 16-element block with its own block scale and its batch's tensor scale
    sp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    sb = synth.loguniform_f32((B * R * K // 16,), 2e-3, 2e-2, seed=35).numpy()
    g = np.array([3e-5, 7e-5], np.float32)
    y, c, e = O.qdq_fwd(sp, x, sb, g, want_codes=True)
    for b in range(B):
        for r in range(R):
            for j in range(K // 16):
                u = (b * R + r) * (K // 16) + j
                ys, cs, es = O.qdq_fwd(sp, x[b:b + 1, r:r + 1, 16 * j:16 * j + 16], sb[u:u + 1],
                                       g[b:b + 1], want_codes=True)
                assert np.array_equal(ys[0, 0], y[b, r, 16 * j:16 * j + 16])
                assert np.array_equal(cs[0, 0], c[b, r, 8 * j:8 * j + 8]) and es[0, 0, 0] == e[b, r, j]


def test_rows_of_eight_times_odd_elements():
    """Rows of K = 8 * odd elements (the library's boundary allows K % 8 == 0):
    per-channel and per-head QDQ and gradients equal the per-element results of
    a K % 16 == 0 layout holding the same rows (zero padding changes no other
    element), codes included; block and group formats reject such K."""
    B, R, K = 2, 5, 24
    x = bits(synth.normal_bf16((B, R, K), 0.02, seed=36))
    dy = bits(synth.normal_bf16((B, R, K), 1.0, seed=37))
    pad = lambda a: np.concatenate([a, np.zeros((B, R, 8), np.uint16)], axis=2)  # K -> 32
    for sp, n in [(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), B * R),
                  (O.spec(O.INT4, O.PER_CHANNEL, qmin=-8, qmax=7), B * R),
                  (O.spec(O.FP8_E4M3, O.PER_HEAD), R)]:
        s = synth.loguniform_f32((n,), 1e-4, 4e-4, seed=38).numpy()
        if sp.fmt == O.INT4:
            s = s * 30
        y, c, _ = O.qdq_fwd(sp, x, s, want_codes=True)
        yp, cp, _ = O.qdq_fwd(sp, pad(x), s, want_codes=True)
        assert np.array_equal(y, yp[:, :, :K])
        assert np.array_equal(c, cp[:, :, :c.shape[2]])
        g = O.scale_grad(sp, x, dy, s)
        gp = O.scale_grad(sp, pad(x), pad(dy), s)
        assert np.array_equal(g["dscale"], gp["dscale"]) and np.array_equal(g["dx"], gp["dx"][:, :, :K])
    for sp in (O.spec(O.NVFP4, O.PER_GROUP, group=16), O.spec(O.INT4, O.PER_GROUP, group=16, qmin=-8, qmax=7)):
        with pytest.raises(ValueError):
            O.qdq_fwd(sp, x, np.ones(B * R * 2, np.float32), np.ones(B, np.float32))
    with pytest.raises(ValueError):  # not a multiple of 8
        O.qdq_fwd(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), x[:, :, :20].copy(),
                  np.ones(B * R, np.float32))


def test_zero_scale_gives_signed_zeros():
    x = bf16_bits_of([1.0, -2.0, 0.0, -0.0] * 4).reshape(1, 1, 16)
    for sp in (O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), O.spec(O.FP8_E4M3, O.PER_TENSOR)):
        y, _, _ = O.qdq_fwd(sp, x, np.zeros(1, np.float32))
        # integer codes have no signed zero; E4M3 codes keep x's sign
        want = x & np.uint16(0x8000) if sp.fmt == O.FP8_E4M3 else np.zeros_like(x)
        assert np.array_equal(y, want)
        g = O.scale_grad(sp, x, x, np.zeros(1, np.float32))
        assert g["dscale"][0] == 0.0
    sp = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    y, _, blk = O.qdq_fwd(sp, x, np.ones(1, np.float32), np.zeros(1, np.float32), want_codes=True)
    assert np.array_equal(y, x & np.uint16(0x8000)) and blk[0, 0, 0] == 0


# --------------------------------------------------------------------------------------
# gradient
# --------------------------------------------------------------------------------------

def test_grad_closed_form_single_elements():
    sp = O.spec(O.INT8, O.PER_TENSOR, qmin=-128, qmax=127)
    cases = [  # (x, s, dy, expected dS)
        (2.296875, 1.0, 1.0, 2 - 2.296875),      # in range: q - v
        (200.0, 1.0, 2.0, 2 * 127.0),            # clamped high: q = qmax
        (127.0, 1.0, 1.0, 127.0),                # at the bound counts as clamped
        (-128.0, 1.0, 1.0, -128.0),
        (-127.5, 1.0, 1.0, -128 + 127.5),        # inside: rounds to -128 (even)
        (0.375, 0.25, -3.0, -3.0 * (2 - 1.5)),
    ]
    for x, s, dy, want in cases:
        xb = np.tile(bf16_bits_of([x]), 16).reshape(1, 1, 16)
        xb[0, 0, 1:] = 0
        dyb = np.tile(bf16_bits_of([dy]), 16).reshape(1, 1, 16)
        g = O.scale_grad(sp, xb, dyb, np.array([s], np.float32))
        assert g["dscale"][0] == want, (x, s, g["dscale"][0], want)
    sp = O.spec(O.FP8_E4M3, O.PER_TENSOR)
    xb = np.zeros((1, 1, 16), np.uint16)
    xb[0, 0, 0] = bf16_bits_of([500.0])[0]
    dyb = np.tile(bf16_bits_of([1.0]), 16).reshape(1, 1, 16)
    assert O.scale_grad(sp, xb, dyb, np.ones(1, np.float32))["dscale"][0] == 448.0


def test_int8_grad_matches_torch_learnable_fake_quant():
    """torch._fake_quantize_learnable_per_channel_affine (grad_factor 1) gives
    the same straight-through scale gradient where no |v| sits within half a
    step of the clamp bounds (torch masks on the rounded value, the LSQ form on
    the unrounded one; elsewhere the two definitions coincide)."""
    N, K = 32, 512
    w = synth.normal_bf16((N, K), 0.02, seed=41)
    s = synth.loguniform_f32((N,), 1.2e-4, 4e-4, seed=42)
    v = w.float() / s[:, None]
    near = ((v.abs() - 127.0).abs() < 0.75) | ((v + 128).abs() < 0.75)
    w = torch.where(near, torch.zeros_like(w), w)
    dy = synth.normal_bf16((N, K), 1.0, seed=43)
    xs = w.float().requires_grad_(True)
    sc = s.clone().requires_grad_(True)
    zp = torch.zeros(N, dtype=torch.float32, requires_grad=True)
    out = torch._fake_quantize_learnable_per_channel_affine(xs, sc, zp, 0, -128, 127, 1.0)
    out.backward(dy.float())
    gr = O.scale_grad(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), bits(w)[None],
                      bits(dy)[None], s.numpy())
    err = np.abs(gr["dscale"] - sc.grad.double().numpy())
    assert np.all(err <= 2e-5 * gr["dscale_abs"]), err.max()
    assert np.array_equal(f32_of_bits(gr["dx"][0]), xs.grad.numpy())


def test_grad_shard_merge_and_granularity_consistency():
    B, R, K = 2, 16, 256
    x = bits(synth.normal_bf16((B, R, K), 0.02, seed=44))
    dy = bits(synth.normal_bf16((B, R, K), 1.0, seed=45))
    s = synth.loguniform_f32((1,), 1e-4, 2e-4, seed=46).numpy()
    ch = O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127)
    tn = O.spec(O.INT8, O.PER_TENSOR, qmin=-128, qmax=127)
    hd = O.spec(O.INT8, O.PER_HEAD, qmin=-128, qmax=127)
    g_ch = O.scale_grad(ch, x, dy, np.full(B * R, s[0], np.float32))["dscale"]
    g_tn = O.scale_grad(tn, x, dy, np.full(B, s[0], np.float32))["dscale"]
    g_hd = O.scale_grad(hd, x, dy, np.full(R, s[0], np.float32))["dscale"]
    assert np.allclose(g_tn, g_ch.reshape(B, R).sum(1), rtol=1e-12, atol=1e-12)
    assert np.allclose(g_hd, g_ch.reshape(B, R).sum(0), rtol=1e-12, atol=1e-12)
    # K split into two shards with the same per-channel scale
    sc = np.full(B * R, s[0], np.float32)
    a = O.scale_grad(ch, x[..., :128], dy[..., :128], sc)["dscale"]
    b = O.scale_grad(ch, x[..., 128:], dy[..., 128:], sc)["dscale"]
    assert np.allclose(a + b, g_ch, rtol=1e-12, atol=1e-12)


def test_nvfp4_dynamic_tensor_grad_is_block_grads_weighted_by_block_codes():
    """With the block scale fixed to its dynamic value, the tensor-scale
    gradient is sum_b dec(e_b) * (learned-mode block gradient)."""
    B, R, K = 2, 8, 64
    x = bits(synth.normal_outliers_bf16((B, R, K), 1.0, 1e-2, 30.0, seed=47))
    dy = bits(synth.normal_bf16((B, R, K), 1.0, seed=48))
    g = np.array([1.0 / 2688, 0.02 / 2688], np.float32)
    dyn = O.spec(O.NVFP4, O.PER_GROUP, group=16, mode=O.SCALE_DYNAMIC_BLOCK)
    lrn = O.spec(O.NVFP4, O.PER_GROUP, group=16)
    amax = np.abs(f32_of_bits(x).reshape(-1, 16)).max(1).astype(np.float64)
    sb = (amax / 6.0).astype(np.float32)  # the dynamic block scale, fl32(amax / 6)
    y_d, _, blk_d = O.qdq_fwd(dyn, x, None, g, want_codes=True)
    y_l, _, blk_l = O.qdq_fwd(lrn, x, sb, g, want_codes=True)
    assert np.array_equal(y_d, y_l) and np.array_equal(blk_d, blk_l)
    gd = O.scale_grad(dyn, x, dy, None, g)
    gl = O.scale_grad(lrn, x, dy, sb, g)
    dec = np.array([O.e4m3_decode(c) for c in blk_l.reshape(-1)])
    want = (dec * gl["dscale"]).reshape(B, -1).sum(1)
    assert np.allclose(gd["dtensor_scale"], want, rtol=1e-12, atol=1e-12)
    assert np.array_equal(gd["dx"], gl["dx"])


# --------------------------------------------------------------------------------------
# observer and init
# --------------------------------------------------------------------------------------

def test_observer_matches_numpy_and_merges_exactly():
    x = synth.head_normal_bf16(256, 8, 64, 0.1, 10.0, seed=51)
    xb = bits(x)
    mn, mx = O.observer_minmax(xb)
    xf = x.float().numpy()
    assert np.array_equal(mn, xf.min(axis=(0, 2))) and np.array_equal(mx, xf.max(axis=(0, 2)))
    # running merge over token shards equals one pass over all tokens
    lo, hi = O.observer_minmax(xb[:100])
    lo, hi = O.observer_minmax(xb[100:180], lo, hi)
    lo, hi = O.observer_minmax(xb[180:], lo, hi)
    assert np.array_equal(lo.view(np.uint32), mn.view(np.uint32))
    assert np.array_equal(hi.view(np.uint32), mx.view(np.uint32))
    # each result is an element of its head
    for h in range(8):
        assert mn[h] in xf[:, h, :] and mx[h] in xf[:, h, :]


def test_observer_signed_zero_order():
    x = np.zeros((4, 2, 16), np.uint16)
    x[1, 0, 3] = 0x8000  # head 0 holds +0 and -0 only
    x[:, 1, :] = 0x8000  # head 1 holds -0 only
    mn, mx = O.observer_minmax(x)
    assert math.copysign(1, mn[0]) < 0 and math.copysign(1, mx[0]) > 0
    assert math.copysign(1, mn[1]) < 0 and math.copysign(1, mx[1]) < 0


def test_minmax_scale_closed_form():
    s = O.minmax_scale(np.array([-3.5, -0.0, 1.0], np.float32), np.array([2.0, 0.0, 7.0], np.float32))
    assert s[0] == 2.0 ** -7 and s[1] == 0.0 and s[2] == np.float32(7.0 / 448)


def test_scale_init_closed_forms():
    x = np.zeros((1, 2, 256), np.float32)
    x[0, 0, 5] = -1.75
    x[0, 1, 200] = 0.875
    x[0, 1, 17] = -0.5
    xb = bf16_bits_of(x.reshape(-1)).reshape(1, 2, 256)
    s, _ = O.scale_init(O.spec(O.INT4, O.PER_GROUP, group=128, qmin=-8, qmax=7), xb)
    assert list(s) == [0.25, 0.0, 0.5 / 7, 0.125]
    s, _ = O.scale_init(O.spec(O.INT8, O.PER_CHANNEL, qmin=-128, qmax=127), xb)
    assert list(s) == [np.float32(1.75 / 127), np.float32(0.875 / 127)]
    sb, g = O.scale_init(O.spec(O.NVFP4, O.PER_GROUP, group=16), xb)
    assert g[0] == np.float32(1.75 / 2688)
    assert sb[0] == np.float32(1.75 / 6) and sb[1] == 0 and sb[16 + 1] == np.float32(0.5 / 6)
    _, gd = O.scale_init(O.spec(O.NVFP4, O.PER_GROUP, group=16, mode=O.SCALE_DYNAMIC_BLOCK), xb)
    assert gd[0] == g[0]


def test_grouped_gemm_reference_pins():
    """The oracle's fused-GEMM reference: one-hot rows return rows of w_hat;
    a tiny case equals a brute-force triple loop over the oracle's w_hat."""
    E, N, K = 2, 4, 32
    w = bits(synth.normal_bf16((E, N, K), 0.02, seed=61))
    s = synth.loguniform_f32((E * N * K // 16,), 2e-3, 2e-2, seed=62).numpy()
    g = np.array([3e-5, 6e-5], np.float32)
    wh, _, _ = O.qdq_fwd(O.spec(O.NVFP4, O.PER_GROUP, group=16), w, s, g)
    whf = f32_of_bits(wh).astype(np.float64)
    off = np.array([0, 3, 5])
    x = np.zeros((5, K), np.float32)
    cols = [0, 7, 31, 16, 2]
    x[np.arange(5), cols] = 1.0
    y, a = O.grouped_qdq_gemm(bf16_bits_of(x.reshape(-1)).reshape(5, K), off, w, s, g)
    for m, c in enumerate(cols):
        e = 0 if m < 3 else 1
        assert np.array_equal(y[m], whf[e, :, c])
    xr = f32_of_bits(bits(synth.normal_bf16((5, K), 1.0, seed=63))).astype(np.float64)
    y, a = O.grouped_qdq_gemm(bf16_bits_of(xr.reshape(-1)).reshape(5, K), off, w, s, g)
    for m in range(5):
        e = 0 if m < 3 else 1
        for n in range(N):
            t = [xr[m, k] * whf[e, n, k] for k in range(K)]
            assert abs(y[m, n] - sum(t)) <= 1e-12 * sum(abs(v) for v in t)
            assert abs(a[m, n] - sum(abs(v) for v in t)) <= 1e-12 * a[m, n]
