// aqfq_device.cuh -- device-side building blocks of libaqfq (sm_103a).
//
// One "chunk" is 16 consecutive BF16 elements along K (32 bytes): one 256-bit
// load per operand, one NVFP4 block, 1/8 of an INT4 g128 group.  Every kernel
// maps one lane to one chunk at a time, so loads are perfectly coalesced
// (a warp streams 1 KiB contiguous per operand) and an NVFP4 block's amax and
// gradient sum never leave the lane.  Three chunk layouts (Lay):
//   L_32  16 elements, one 256-bit access per operand (32-byte aligned data)
//   L_16  16 elements, two 128-bit accesses (data only 16-byte aligned)
//   L_8   8 elements, one 128-bit access (rows of K = 8 * odd elements; only
//         per-tensor, per-channel and per-head INT8 / INT4 / FP8 use it)
//
// Rounding steps follow the library's contract (include/aqfq.h):
//   v = x / s        the IEEE binary32 quotient: per chunk one correctly rounded
//                    reciprocal and Markstein's FMA correction per element (see
//                    Divisor); scales outside [2^-125, 2^125] (zero, negative,
//                    extreme) take __fdiv_rn per element (built without fast math)
//   q = grid(v)      integer grid: clamp then round-half-even by the 1.5*2^23
//                    addition trick (exact for |v| < 2^22); E4M3 / E2M1: the
//                    hardware cvt.rn.satfinite conversions
//   x_hat = bf16(q*s) __fmul_rn (never contracted into an FMA), cvt.rn.bf16x2
// The FP grids are symmetric, so their fast paths work on |x| and put the sign
// of x back on the packed outputs (one bit operation per pair of elements).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace aqfq {

constexpr int kThreads = 256;  // threads per CTA for every streaming kernel
constexpr int kChunk = 16;     // elements per lane-chunk (L_32, L_16)

enum Lay { L_32 = 0, L_16 = 1, L_8 = 2 };
// 32-bit words (two BF16 each) of a chunk, and its bytes
template <int L>
struct LayT {
  static constexpr int NW = L == L_8 ? 4 : 8;
  static constexpr int BYTES = NW * 4;
};

enum Fmt { F_INT8 = 0, F_INT4 = 1, F_FP8 = 2, F_NVFP4 = 3 };
enum Gran { G_TENSOR = 0, G_ROW = 1, G_GROUP = 2, G_HEAD = 3 };

// ---------------------------------------------------------------------------
// n / d for 32-bit n by multiply-high and shifts (Granlund & Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994, Fig. 4.1).
// ---------------------------------------------------------------------------
struct FastDiv {
  uint32_t d, m, s1, s2;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;  // l = ceil(log2 d)
  f.m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 1 ? l - 1 : 0;
  return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// ---------------------------------------------------------------------------
// 256-bit streaming memory access (sm_100+ vector width)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_stream(const void* p, uint32_t (&w)[8]) {
  asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
        "=r"(w[7])
      : "l"(p));
}

__device__ __forceinline__ void ld_stream_v4(const void* p, uint32_t& a, uint32_t& b, uint32_t& c,
                                             uint32_t& d) {
  // (the evict-first L2 priority exists only for 256-bit accesses)
  asm("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
      : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
      : "l"(p));
}

__device__ __forceinline__ void st_32(void* p, uint32_t a) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

__device__ __forceinline__ void st_256(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ void st_128(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_64(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// chunk gc of a BF16 tensor in layout L
template <int L>
__device__ __forceinline__ void ld_chunk(const uint8_t* base, uint64_t gc,
                                         uint32_t (&w)[LayT<L>::NW]) {
  const uint8_t* p = base + gc * LayT<L>::BYTES;
  if constexpr (L == L_32) {
    ld_stream(p, w);
  } else {
    ld_stream_v4(p, w[0], w[1], w[2], w[3]);
    if constexpr (L == L_16) ld_stream_v4(p + 16, w[4], w[5], w[6], w[7]);
  }
}

template <int L>
__device__ __forceinline__ void st_chunk(uint8_t* base, uint64_t gc,
                                         const uint32_t (&w)[LayT<L>::NW]) {
  uint8_t* p = base + gc * LayT<L>::BYTES;
  if constexpr (L == L_32) {
    st_256(p, w);
  } else {
    st_128(p, w[0], w[1], w[2], w[3]);
    if constexpr (L == L_16) st_128(p + 16, w[4], w[5], w[6], w[7]);
  }
}

// packed codes of chunk gc: INT8 / FP8 one byte per element, INT4 / NVFP4 one
// nibble (cw holds them in order, element 0 lowest)
template <int L, bool BYTE_CODES>
__device__ __forceinline__ void st_codes(uint8_t* codes, uint64_t gc, const uint32_t (&cw)[4]) {
  if constexpr (L == L_8) {
    if constexpr (BYTE_CODES) st_64(codes + gc * 8, cw[0], cw[1]);
    else st_32(codes + gc * 4, cw[0]);
  } else {
    if constexpr (BYTE_CODES) st_128(codes + gc * 16, cw[0], cw[1], cw[2], cw[3]);
    else st_64(codes + gc * 8, cw[0], cw[1]);
  }
}

// ---------------------------------------------------------------------------
// BF16 <-> binary32
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// two binary32 values -> packed BF16 pair, round to nearest even (hi in bits 31..16)
__device__ __forceinline__ uint32_t pack_bf16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// Pairs of binary32 values in one 64-bit register (element 2i in the low
// half) for the packed f32x2 instructions of sm_100-class GPUs.  Each lane is
// rounded to nearest even as the scalar instruction rounds it (no flush of
// subnormals), so a packed step gives the bits of two scalar steps.
// ---------------------------------------------------------------------------
typedef unsigned long long f2;
__device__ __forceinline__ f2 mk2(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo2(f2 v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float hi2(f2 v) { return __uint_as_float(uint32_t(v >> 32)); }
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// a BF16 pair (element 2i in the low half) as two binary32 values (exact)
__device__ __forceinline__ f2 bf2(uint32_t w) { return mk2(bf_lo(w), bf_hi(w)); }
// both lanes rounded to a BF16 pair, lane 0 in bits 15..0
__device__ __forceinline__ uint32_t pack2(f2 v) { return pack_bf16x2(hi2(v), lo2(v)); }

__device__ __forceinline__ float sign_zero(float x) {
  return __uint_as_float(__float_as_uint(x) & 0x80000000u);
}

// ---------------------------------------------------------------------------
// E4M3 and E2M1 conversions (PTX cvt, saturating to the largest finite value)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float h2f(uint16_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}

// packed E4M3 pair (element in bits 7..0 -> .x) -> two binary32 values (exact)
__device__ __forceinline__ float2 dec_e4m3x2(uint32_t c) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)c));
  return make_float2(h2f((uint16_t)(h & 0xFFFF)), h2f((uint16_t)(h >> 16)));
}

__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 t, z;\n\t"
      "mov.b16 {t, z}, 0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "mov.b32 %0, {t, z, z, z}; }"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// packed E2M1 pair (element in bits 3..0 -> .x) -> two binary32 values (exact)
__device__ __forceinline__ float2 dec_e2m1x2(uint32_t c) {
  uint32_t h;
  asm("{ .reg .b8 t, u, v, w;\n\t"
      "mov.b32 {t, u, v, w}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t; }"
      : "=r"(h)
      : "r"(c));
  return make_float2(h2f((uint16_t)(h & 0xFFFF)), h2f((uint16_t)(h >> 16)));
}

// ---------------------------------------------------------------------------
// Element grids.  quant_pair rounds (v0, v1) = elements (2i, 2i+1) of a chunk
// and returns the grid values, the packed codes of the pair and whether the
// clamp is active for each (the gradient's switch).
// ---------------------------------------------------------------------------
struct IntRange {
  float qmin, qmax;
  // With `centred`, c = (qmin + qmax) / 2 and h = (qmax - qmin) / 2 decide
  // the clamp in one comparison: |RN(v - c)| >= h exactly when v <= qmin or
  // v >= qmax, for every binary32 v (NaN: neither).  The forward ignores them.
  float c = 0.0f, h = 0.0f;
  bool centred = false;
};

// An integer grid [qmin, qmax] (integers, qmin < qmax) with its one-compare
// clamp test where that test is exact: c = 0, or c = -1/2 with qmax not a
// power of two, or c = +1/2 with -qmin not a power of two, and h >= 1.
// v - c is then exact wherever it lies within rounding distance of h (it
// lands in v's binade or a finer one); with c = -1/2 and qmax = 2^k, v just
// below qmax has a finer ulp than v + 1/2, which can round up onto h (qmax = 1,
// v = 1 - 2^-24).  Checked against the two comparisons on all 2^32 binary32
// values for [-8,7], [-128,127], [-127,127], [-7,7], [-4,3], [-3,4], [-16,16]
// (and the two excluded cases [-2,1], [-1,2], one mismatch each).
inline IntRange int_range(float qmin, float qmax) {
  IntRange r;
  r.qmin = qmin;
  r.qmax = qmax;
  r.c = 0.5f * (qmin + qmax);  // exact: integers of magnitude <= 2^22
  r.h = 0.5f * (qmax - qmin);
  auto pow2 = [](float x) {
    const long long q = (long long)x;
    return x >= 1.0f && float(q) == x && (q & (q - 1)) == 0;
  };
  const bool ok = r.c == 0.0f || (r.c == -0.5f && !pow2(qmax)) || (r.c == 0.5f && !pow2(-qmin));
  r.centred = ok && r.h >= 1.0f;
  return r;
}

// clamp then round half to even via t = vc + 1.5*2^23 (|vc| <= 128 << 2^22):
// t's low bits hold the integer in two's complement; t - 1.5*2^23 is the
// integer as +0 for zero (an integer code carries no sign).
__device__ __forceinline__ float int_round(float v, const IntRange& r, uint32_t& code) {
  const float kMagic = 12582912.0f;  // 1.5 * 2^23
  float vc = fminf(fmaxf(v, r.qmin), r.qmax);
  float t = __fadd_rn(vc, kMagic);
  code = __float_as_uint(t);
  return __fsub_rn(t, kMagic);
}

// int_round of both lanes of a pair; t receives the biased sums (the codes in
// their low bits)
__device__ __forceinline__ f2 int_round2(f2 v, const IntRange& r, f2& t) {
  const f2 kMagic = mk2(12582912.0f, 12582912.0f);  // 1.5 * 2^23
  const f2 vc = mk2(fminf(fmaxf(lo2(v), r.qmin), r.qmax), fminf(fmaxf(hi2(v), r.qmin), r.qmax));
  t = add2(vc, kMagic);
  return sub2(t, kMagic);
}

template <int FMT>
__device__ __forceinline__ uint32_t int_codes(f2 t) {
  const uint32_t c0 = __float_as_uint(lo2(t)), c1 = __float_as_uint(hi2(t));
  if constexpr (FMT == F_INT8) return (c0 & 0xFFu) | ((c1 & 0xFFu) << 8);
  else return (c0 & 0xFu) | ((c1 & 0xFu) << 4);
}

template <int FMT>
__device__ __forceinline__ void quant_pair(float v0, float v1, const IntRange& r, float& q0,
                                           float& q1, uint32_t& code, bool& k0, bool& k1) {
  if constexpr (FMT == F_INT8 || FMT == F_INT4) {
    uint32_t c0, c1;
    q0 = int_round(v0, r, c0);
    q1 = int_round(v1, r, c1);
    if constexpr (FMT == F_INT8) code = (c0 & 0xFFu) | ((c1 & 0xFFu) << 8);
    else code = (c0 & 0xFu) | ((c1 & 0xFu) << 4);
    k0 = (v0 <= r.qmin) || (v0 >= r.qmax);
    k1 = (v1 <= r.qmin) || (v1 >= r.qmax);
  } else if constexpr (FMT == F_FP8) {
    code = cvt_e4m3x2(v1, v0);
    float2 d = dec_e4m3x2(code);
    q0 = d.x;
    q1 = d.y;
    k0 = fabsf(v0) >= 448.0f;
    k1 = fabsf(v1) >= 448.0f;
  } else {
    code = cvt_e2m1x2(v1, v0);
    float2 d = dec_e2m1x2(code);
    q0 = d.x;
    q1 = d.y;
    k0 = fabsf(v0) >= 6.0f;
    k1 = fabsf(v1) >= 6.0f;
  }
}

// bits of the packed codes of one chunk: INT8/FP8 one byte per element (16 B),
// INT4/NVFP4 one nibble per element (8 B)
template <int FMT>
__device__ __forceinline__ void put_code(uint32_t (&cw)[4], int pair, uint32_t code) {
  if constexpr (FMT == F_INT8 || FMT == F_FP8) {
    cw[pair >> 1] |= code << (16 * (pair & 1));
  } else {
    cw[pair >> 2] |= code << (8 * (pair & 3));
  }
}

// ---------------------------------------------------------------------------
// NVFP4 block scale: e = E4M3(S_b / g) (saturating), S_hat = dec(e) * g
// ---------------------------------------------------------------------------
__device__ __forceinline__ float nvfp4_block_scale(float sb, float g, uint32_t& ecode) {
  float r = (g != 0.0f) ? __fdiv_rn(sb, g) : 0.0f;
  ecode = cvt_e4m3x2(0.0f, r) & 0xFFu;
  return __fmul_rn(dec_e4m3x2(ecode).x, g);
}

// largest |x| of a chunk as binary32 (exact: a BF16 value)
template <int NW>
__device__ __forceinline__ float chunk_amax(const uint32_t (&w)[NW]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  uint32_t a = max(m & 0xFFFFu, m >> 16);
  return __uint_as_float(a << 16);
}

// E2M1 / E4M3 rounding of a pair followed by the exact decode: returns the
// packed f16 pair of grid values (element lo -> bits 15..0); the *c forms also
// return the codes (E2M1: byte, lo in bits 3..0; E4M3: 16 bits, lo in 7..0)
__device__ __forceinline__ uint32_t e2m1_q2(float hi, float lo) {
  uint32_t h;
  asm("{ .reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t; }"
      : "=r"(h)
      : "f"(hi), "f"(lo));
  return h;
}

__device__ __forceinline__ uint32_t e2m1_q2c(float hi, float lo, uint32_t& code) {
  uint32_t h, c;
  asm("{ .reg .b8 t, z;\n\t"
      "mov.b16 {t, z}, 0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %3;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t"
      "mov.b32 %1, {t, z, z, z}; }"
      : "=r"(h), "=r"(c)
      : "f"(hi), "f"(lo));
  code = c;
  return h;
}

__device__ __forceinline__ uint32_t e4m3_q2(float hi, float lo) {
  uint32_t h;
  asm("{ .reg .b16 t;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, t; }"
      : "=r"(h)
      : "f"(hi), "f"(lo));
  return h;
}

__device__ __forceinline__ uint32_t e4m3_q2c(float hi, float lo, uint32_t& code) {
  uint32_t h;
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %1, %2, %3;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, %1;"
      : "=r"(h), "=h"(c)
      : "f"(hi), "f"(lo));
  code = c;
  return h;
}

template <int FMT>
__device__ __forceinline__ uint32_t fp_q2(float hi, float lo) {
  if constexpr (FMT == F_FP8) return e4m3_q2(hi, lo);
  else return e2m1_q2(hi, lo);
}

template <int FMT>
__device__ __forceinline__ uint32_t fp_q2c(float hi, float lo, uint32_t& code) {
  if constexpr (FMT == F_FP8) return e4m3_q2c(hi, lo, code);
  else return e2m1_q2c(hi, lo, code);
}

// q - m with q an f16 grid value and m binary32 (mixed-precision subtract)
__device__ __forceinline__ float sub_h_f(uint16_t q, float m) {
  float d;
  asm("sub.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(q), "f"(m));
  return d;
}

// ---------------------------------------------------------------------------
// Division by a chunk's scale s.
// When 2^-64 <= s <= 2^64 and the chunk's largest |x| / s stays below 2^100:
// r = RN(1/s) once per chunk, then per element Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
//   q0 = RN(x * r),  e = RN(x - q0 * s) (one FMA),  v = RN(q0 + e * r).
// No step can overflow.  e is exact whenever |x| >= 2^-102 (its quantum is at
// least that of q0 * s, which stays above 2^-149), and then v is the IEEE
// quotient x / s unless that quotient is below 2^-126.  So v can differ from
// the IEEE quotient only when |x / s| < 2^-38 (|x| < 2^-102 with s >= 2^-64,
// or a subnormal quotient), by at most two units in the last place, and every
// grid maps such quotients to zero: no code or dequantised value changes; a
// gradient term changes by at most two ulps of itself.  (Checked on the GPU
// against __fdiv_rn: every BF16 mantissa against every binary32 mantissa of s
// at six exponent pairs, and every BF16 x against 2^18 random s in range:
// no difference at |x / s| >= 2^-38.)  With x = -0 the steps give +0; the
// forward therefore divides |x| and puts the sign back itself.
// The forward checks the chunk's largest |x| before taking the fast path.
// The gradient does not: a quotient beyond binary32 range makes q0 infinite
// and v NaN, the NaN reaches the chunk's gradient sum, and the chunk is then
// recomputed with IEEE division; finite inputs give no NaN otherwise.
// Chunks outside these bounds take __fdiv_rn per element.
// ---------------------------------------------------------------------------
struct Divisor {
  float s, r;
  bool fast;
};

__device__ __forceinline__ Divisor make_divisor(float s) {
  Divisor d;
  d.s = s;
  d.r = __frcp_rn(s);
  d.fast = (s >= 0x1p-64f) && (s <= 0x1p64f);
  return d;
}

// forward: also require the chunk's largest |x| (exact) / s <= 2^100
__device__ __forceinline__ Divisor make_divisor(float s, float amax) {
  Divisor d = make_divisor(s);
  d.fast = d.fast && (__fmul_rn(amax, d.r) <= 0x1p100f);
  return d;
}

__device__ __forceinline__ float mdiv(float x, const Divisor& d) {
  const float q0 = __fmul_rn(x, d.r);
  const float e = __fmaf_rn(-q0, d.s, x);
  return __fmaf_rn(e, d.r, q0);
}

// mdiv of both lanes of a pair (q0 (-s) + x is the same exact value as
// (-q0) s + x, so every lane has mdiv's bits)
__device__ __forceinline__ f2 mdiv2(f2 x, const Divisor& d) {
  const f2 r = mk2(d.r, d.r);
  const f2 q0 = mul2(x, r);
  const f2 e = fma2(q0, mk2(-d.s, -d.s), x);
  return fma2(e, r, q0);
}

// The sum of a chunk's 2 NW gradient terms in one fixed order, shared by the
// fast and the IEEE paths: a pairwise tree over the pairs, lane by lane (the
// even elements' and the odd elements' totals), then their sum.  log2(2 NW)
// levels of rounding, as a pairwise tree over the elements.
template <int NW>
__device__ __forceinline__ float chunk_sum(f2 (&t)[NW]) {
  static_assert(NW >= 1 && (NW & (NW - 1)) == 0, "a power of two");
#pragma unroll
  for (int w = 1; w < NW; w *= 2) {
#pragma unroll
    for (int i = 0; i < NW; i += 2 * w) t[i] = add2(t[i], t[i + w]);
  }
  return __fadd_rn(lo2(t[0]), hi2(t[0]));
}

// ---------------------------------------------------------------------------
// Fast-path chunks (Divisor::fast)
// ---------------------------------------------------------------------------
template <int FMT>
constexpr float grid_max() {
  return FMT == F_FP8 ? 448.0f : 6.0f;
}

// sign bits of the two elements of a BF16 pair moved to their code positions
template <int FMT>
__device__ __forceinline__ uint32_t code_signs(uint32_t sgn) {
  if constexpr (FMT == F_FP8) return ((sgn >> 8) & 0x80u) | ((sgn >> 16) & 0x8000u);
  else return ((sgn >> 12) & 0x8u) | ((sgn >> 24) & 0x80u);
}

template <int FMT, bool CODES, int NW>
__device__ __forceinline__ void qdq_chunk_fast(const uint32_t (&xw)[NW], const Divisor& d,
                                               const IntRange& r, uint32_t (&yw)[NW],
                                               uint32_t (&cw)[4]) {
  if (CODES) cw[0] = cw[1] = cw[2] = cw[3] = 0;
  const f2 S2 = mk2(d.s, d.s);
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    uint32_t code = 0;
    if constexpr (FMT == F_INT8 || FMT == F_INT4) {
      // the integer grid maps +-0 alike (an integer code has no sign)
      f2 t;
      const f2 q = int_round2(mdiv2(bf2(xw[i]), d), r, t);
      if (CODES) code = int_codes<FMT>(t);
      yw[i] = pack2(mul2(q, S2));
    } else {
      // symmetric grid: round |v|, then give x's sign to the value and the code
      const f2 a = mdiv2(bf2(xw[i] & 0x7FFF7FFFu), d);
      const uint32_t h = CODES ? fp_q2c<FMT>(hi2(a), lo2(a), code) : fp_q2<FMT>(hi2(a), lo2(a));
      const uint32_t sgn = xw[i] & 0x80008000u;
      yw[i] = pack2(mul2(mk2(h2f((uint16_t)(h & 0xFFFFu)), h2f((uint16_t)(h >> 16))), S2)) | sgn;
      if (CODES) code |= code_signs<FMT>(sgn);
    }
    if (CODES) put_code<FMT>(cw, i, code);
  }
}

// FWD: also the forward's x_hat of the chunk into yw (the same bits as
// qdq_chunk_fast: FP grids give |q| * s the sign of x, so -0 stays -0).
// CENT: integer grids decide the clamp by |v - c| >= h (IntRange::centred).
template <int FMT, bool DX, bool FWD, bool CENT, int NW>
__device__ __forceinline__ float grad_chunk_fast_impl(const uint32_t (&xw)[NW],
                                                      const uint32_t (&dw)[NW], const Divisor& d,
                                                      const IntRange& r, uint32_t (&dxw)[NW],
                                                      uint32_t* yw) {
  f2 t[NW];
  const f2 S2 = mk2(d.s, d.s);
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    // the sign of a zero quotient does not change a gradient term
    const f2 v = mdiv2(bf2(xw[i]), d);
    const float v0 = lo2(v), v1 = hi2(v);
    bool k0, k1;
    f2 term;
    if constexpr (FMT == F_INT8 || FMT == F_INT4) {
      f2 tb;
      const f2 q = int_round2(v, r, tb);
      if constexpr (CENT) {
        const f2 vc = sub2(v, mk2(r.c, r.c));
        k0 = fabsf(lo2(vc)) >= r.h;
        k1 = fabsf(hi2(vc)) >= r.h;
      } else {
        k0 = (v0 <= r.qmin) || (v0 >= r.qmax);
        k1 = (v1 <= r.qmin) || (v1 >= r.qmax);
      }
      const f2 dq = sub2(q, v);
      term = mk2(k0 ? lo2(q) : lo2(dq), k1 ? hi2(q) : hi2(dq));
      if constexpr (FWD) yw[i] = pack2(mul2(q, S2));
    } else {
      const uint32_t h = fp_q2<FMT>(v1, v0);
      k0 = fabsf(v0) >= grid_max<FMT>();
      k1 = fabsf(v1) >= grid_max<FMT>();
      term = mk2(sub_h_f((uint16_t)(h & 0xFFFFu), k0 ? 0.0f : v0),
                 sub_h_f((uint16_t)(h >> 16), k1 ? 0.0f : v1));
      if constexpr (FWD) {
        const uint32_t a = h & 0x7FFF7FFFu;  // |q| of the pair (f16)
        yw[i] = pack2(mul2(mk2(h2f((uint16_t)(a & 0xFFFFu)), h2f((uint16_t)(a >> 16))), S2)) |
                (xw[i] & 0x80008000u);
      }
    }
    t[i] = mul2(bf2(dw[i]), term);
    if (DX) dxw[i] = (k0 ? 0u : (dw[i] & 0xFFFFu)) | (k1 ? 0u : (dw[i] & 0xFFFF0000u));
  }
  return chunk_sum(t);
}

template <int FMT, bool DX, bool FWD = false, int NW>
__device__ __forceinline__ float grad_chunk_fast(const uint32_t (&xw)[NW], const uint32_t (&dw)[NW],
                                                 const Divisor& d, const IntRange& r,
                                                 uint32_t (&dxw)[NW], uint32_t* yw = nullptr) {
  if constexpr (FMT == F_INT8 || FMT == F_INT4) {
    if (r.centred) return grad_chunk_fast_impl<FMT, DX, FWD, true>(xw, dw, d, r, dxw, yw);
  }
  return grad_chunk_fast_impl<FMT, DX, FWD, false>(xw, dw, d, r, dxw, yw);
}

// ---------------------------------------------------------------------------
// One chunk, forward, IEEE division per element (any scale; only chunks
// outside the fast path's bounds come here): y = bf16(q * s)
// ---------------------------------------------------------------------------
template <int FMT, bool CODES, int NW>
__device__ __forceinline__ void qdq_chunk(const uint32_t (&xw)[NW], float s, const IntRange& r,
                                          uint32_t (&yw)[NW], uint32_t (&cw)[4]) {
  if (CODES) cw[0] = cw[1] = cw[2] = cw[3] = 0;
  const bool zero = (s == 0.0f);
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const float x0 = bf_lo(xw[i]), x1 = bf_hi(xw[i]);
    const float v0 = zero ? sign_zero(x0) : __fdiv_rn(x0, s);
    const float v1 = zero ? sign_zero(x1) : __fdiv_rn(x1, s);
    float q0, q1;
    uint32_t code;
    bool k0, k1;
    quant_pair<FMT>(v0, v1, r, q0, q1, code, k0, k1);
    yw[i] = pack_bf16x2(__fmul_rn(q1, s), __fmul_rn(q0, s));
    if (CODES) put_code<FMT>(cw, i, code);
  }
}

// ---------------------------------------------------------------------------
// One chunk, backward, IEEE division per element (as above):
// returns sum_i dy_i * (clamped ? q_i : q_i - v_i), summed in chunk_sum's
// fixed order; optional STE mask of dy.  The term q - v is exact
// in binary32 (q and v are within a factor of two, Sterbenz), so the only
// roundings are one per product and four levels of the sum.
// ---------------------------------------------------------------------------
template <int FMT, bool DX, int NW>
__device__ __forceinline__ float grad_chunk(const uint32_t (&xw)[NW], const uint32_t (&dw)[NW],
                                            float s, const IntRange& r, uint32_t (&dxw)[NW]) {
  f2 t[NW];
  const bool zero = (s == 0.0f);
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const float x0 = bf_lo(xw[i]), x1 = bf_hi(xw[i]);
    const float v0 = zero ? sign_zero(x0) : __fdiv_rn(x0, s);
    const float v1 = zero ? sign_zero(x1) : __fdiv_rn(x1, s);
    float q0, q1;
    uint32_t code;
    bool k0, k1;
    quant_pair<FMT>(v0, v1, r, q0, q1, code, k0, k1);
    const float term0 = k0 ? q0 : __fsub_rn(q0, v0);
    const float term1 = k1 ? q1 : __fsub_rn(q1, v1);
    t[i] = mul2(bf2(dw[i]), mk2(term0, term1));
    if (DX) dxw[i] = (k0 ? 0u : (dw[i] & 0xFFFFu)) | (k1 ? 0u : (dw[i] & 0xFFFF0000u));
  }
  return chunk_sum(t);
}

}  // namespace aqfq
