/*
 * aqfq_oracle.c -- plain double-precision CPU oracle for learnable-scale
 * fake-quant (TEST INFRASTRUCTURE: only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; it shares no code with the CUDA
 * library).  See aqfq_oracle.h for the layouts and the passages followed.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast
 * math: every rounding below is the one written in the source).
 * OpenMP only splits independent units (rows) across threads; the
 * arithmetic inside a unit is the same as the serial loop.
 */
#include "aqfq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* threads for the parallel loops that follow (timing a single-thread baseline) */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : 1);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------- */
/* binary32 and bf16                                                          */
/* ------------------------------------------------------------------------- */

/* Round a double to binary32, round-to-nearest-even (the C conversion in the
 * default rounding mode).  For the quotient or product of two binary32 values
 * computed exactly or in double this is the correctly rounded binary32 result
 * (53 >= 2*24 + 2, so the double rounding is innocuous). */
static float fl32(double d) { return (float)d; }

float orc_div32(float a, float b) { return fl32((double)a / (double)b); }

/* bf16 is the upper half of a binary32 encoding: 1 sign bit, 8 exponent bits,
 * 7 stored fraction bits (8 significand bits). */
float orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Nearest bf16 value to a binary32 value, ties to the even significand.
 * Written from the format: significand spacing 2^(E-7) for a value in
 * [2^E, 2^(E+1)), fixed at 2^-133 below the normal range; overflow to inf. */
uint16_t orc_bf16_round(float f) {
  uint32_t fu;
  memcpy(&fu, &f, sizeof fu);
  uint16_t sign = (uint16_t)((fu >> 16) & 0x8000u);
  double a = fabs((double)f);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  if (isnan(a)) return (uint16_t)(sign | 0x7FC0u);
  int e;
  frexp(a, &e);               /* a in [2^(e-1), 2^e) */
  int lead = e - 1;
  if (lead < -126) lead = -126;
  double spacing = ldexp(1.0, lead - 7);
  double r = nearbyint(a / spacing) * spacing; /* a/spacing is exact */
  if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
  float rf = (float)r;        /* exact: r has at most 8 significant bits */
  uint32_t ru;
  memcpy(&ru, &rf, sizeof ru);
  return (uint16_t)(sign | (uint16_t)(ru >> 16));
}

/* ------------------------------------------------------------------------- */
/* Element grids (OCP microscaling formats)                                    */
/* ------------------------------------------------------------------------- */

/* E4M3 "fn": sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
 * S.1111.111 is NaN.  Largest finite 448, smallest subnormal 2^-9. */
double orc_e4m3_decode(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 0xF, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp(m / 8.0, 1 - 7) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; values
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives. */
double orc_e2m1_decode(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? (m / 2.0) : ldexp(1.0 + m / 2.0, e - 1);
  return s ? -mag : mag;
}

/* Nearest non-negative code to a >= 0 by trying every finite non-negative code
 * 0..maxcode (their values increase with the code).  On equal distance the
 * even code (last mantissa bit 0) wins.  The distances to the two codes that
 * bracket a are exact in double, so ties are detected exactly. */
static int nearest_code(double a, double (*dec)(int), int maxcode) {
  int best = 0;
  double bestd = fabs(dec(0) - a);
  for (int c = 1; c <= maxcode; ++c) {
    double d = fabs(dec(c) - a);
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return best;
}

/* Saturating ("satfinite") conversion: magnitudes at or above the largest
 * finite value give it; the sign bit follows v, so -0 and small negative
 * values give the negative-zero code. */
int orc_e4m3_encode(double v) {
  int sign = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  return sign | nearest_code(a, orc_e4m3_decode, 0x7E);
}

int orc_e2m1_encode(double v) {
  int sign = signbit(v) ? 0x8 : 0;
  double a = fabs(v);
  if (a >= 6.0) return sign | 0x7;
  return sign | nearest_code(a, orc_e2m1_decode, 0x7);
}

/* Integer grid: round half to even, then clamp to [qmin, qmax]. */
double orc_int_round(double v, int qmin, int qmax) {
  double q = nearbyint(v);
  if (q < (double)qmin) q = (double)qmin;
  if (q > (double)qmax) q = (double)qmax;
  return q;
}

/* ------------------------------------------------------------------------- */
/* One element: v = x / s in binary32, q on the grid, x_hat = bf16(fl32(q*s)) */
/* ------------------------------------------------------------------------- */

typedef struct {
  float v;      /* the binary32 quotient */
  double q;     /* grid value */
  int code;     /* grid code (INT: the integer) */
  int clipped;  /* v at or beyond the grid's end (the clamp is active) */
} orc_elem;

/* fmt here is the element grid: ORC_INT8 / ORC_INT4 (integers in [qmin,qmax]),
 * ORC_FP8_E4M3, ORC_NVFP4 (E2M1 elements). */
static orc_elem quant_elem(int fmt, int qmin, int qmax, float x, float s) {
  orc_elem o;
  /* A zero scale has no quotient; the element is taken as a zero of x's sign
   * (so the output is a signed zero and the gradient term is zero). */
  o.v = (s != 0.0f) ? fl32((double)x / (double)s) : copysignf(0.0f, x);
  if (fmt == ORC_FP8_E4M3) {
    o.code = orc_e4m3_encode(o.v);
    o.q = orc_e4m3_decode(o.code);
    o.clipped = fabs((double)o.v) >= 448.0;
  } else if (fmt == ORC_NVFP4) {
    o.code = orc_e2m1_encode(o.v);
    o.q = orc_e2m1_decode(o.code);
    o.clipped = fabs((double)o.v) >= 6.0;
  } else {
    /* the integer code has no signed zero: dequantisation is code * s */
    o.code = (int)orc_int_round(o.v, qmin, qmax);
    o.q = (double)o.code;
    o.clipped = ((double)o.v <= (double)qmin) || ((double)o.v >= (double)qmax);
  }
  return o;
}

static uint16_t dequant(double q, float s) { return orc_bf16_round(fl32(q * (double)s)); }

/* NVFP4 block scale: E4M3 code of fl32(S_b / g), dequantised scale
 * fl32(dec(code) * g).  A zero tensor scale gives the zero code. */
static float nvfp4_block_scale(float sb, float g, int* ecode) {
  float r = (g != 0.0f) ? fl32((double)sb / (double)g) : 0.0f;
  int e = orc_e4m3_encode(r);
  *ecode = e;
  return fl32(orc_e4m3_decode(e) * (double)g);
}

/* ------------------------------------------------------------------------- */
/* Validation                                                                 */
/* ------------------------------------------------------------------------- */

/* Rows are whole multiples of 8 elements (the library's boundary); the NVFP4
   block and every group (16 elements or more) need K to be a multiple of
   their size. */
static int spec_ok(const orc_spec* sp, int64_t K) {
  if (!sp) return 0;
  if (K % 8 != 0) return 0;
  if (sp->fmt == ORC_NVFP4) {
    return K % 16 == 0 && sp->gran == ORC_PER_GROUP && sp->group == 16 &&
           (sp->mode == ORC_SCALE_LEARNED || sp->mode == ORC_SCALE_DYNAMIC_BLOCK);
  }
  if (sp->mode != ORC_SCALE_LEARNED) return 0;
  if (sp->fmt == ORC_INT8 && !(sp->qmin >= -128 && sp->qmax <= 127 && sp->qmin < 0 && sp->qmax > 0))
    return 0;
  if (sp->fmt == ORC_INT4 && !(sp->qmin >= -8 && sp->qmax <= 7 && sp->qmin < 0 && sp->qmax > 0))
    return 0;
  if (sp->fmt < 0 || sp->fmt > ORC_FP8_E4M3) return 0;
  if (sp->gran == ORC_PER_GROUP)
    return sp->group >= 16 && sp->group % 16 == 0 && K % sp->group == 0;
  return sp->gran == ORC_PER_TENSOR || sp->gran == ORC_PER_CHANNEL || sp->gran == ORC_PER_HEAD;
}

static int64_t scale_index(const orc_spec* sp, int64_t b, int64_t r, int64_t k, int64_t rows,
                           int64_t K) {
  switch (sp->gran) {
    case ORC_PER_TENSOR: return b;
    case ORC_PER_CHANNEL: return b * rows + r;
    case ORC_PER_GROUP: return (b * rows + r) * (K / sp->group) + k / sp->group;
    default: return r; /* ORC_PER_HEAD: one scale per row index, shared over batch */
  }
}

/* ------------------------------------------------------------------------- */
/* Forward                                                                    */
/* ------------------------------------------------------------------------- */

int orc_qdq_fwd(const orc_spec* sp, const uint16_t* x, int64_t batch, int64_t rows, int64_t K,
                const float* scale, const float* tensor_scale, uint16_t* y, uint8_t* codes,
                uint8_t* block_codes) {
  if (!spec_ok(sp, K) || batch < 0 || rows < 0 || !x || !y) return 1;
  const int nvfp4 = sp->fmt == ORC_NVFP4;
  const int dynamic = nvfp4 && sp->mode == ORC_SCALE_DYNAMIC_BLOCK;
  if (nvfp4 && !tensor_scale) return 1;
  if (!dynamic && !scale) return 1;
  const int64_t nrow = batch * rows;
#pragma omp parallel for schedule(static)
  for (int64_t br = 0; br < nrow; ++br) {
    const int64_t b = br / rows, r = br % rows;
    const uint16_t* xr = x + br * K;
    uint16_t* yr = y + br * K;
    if (nvfp4) {
      const float g = tensor_scale[b];
      for (int64_t k0 = 0; k0 < K; k0 += 16) {
        const int64_t blk = br * (K / 16) + k0 / 16;
        float sb;
        if (dynamic) {
          double amax = 0.0;
          for (int i = 0; i < 16; ++i) {
            double a = fabs((double)orc_bf16_value(xr[k0 + i]));
            if (a > amax) amax = a;
          }
          sb = fl32(amax / 6.0);
        } else {
          sb = scale[blk];
        }
        int ecode;
        const float sh = nvfp4_block_scale(sb, g, &ecode);
        if (block_codes) block_codes[blk] = (uint8_t)ecode;
        for (int i = 0; i < 16; ++i) {
          orc_elem o = quant_elem(ORC_NVFP4, 0, 0, orc_bf16_value(xr[k0 + i]), sh);
          yr[k0 + i] = dequant(o.q, sh);
          if (codes) {
            uint8_t* cb = codes + (br * K + k0 + i) / 2;
            if (((k0 + i) & 1) == 0) *cb = (uint8_t)(o.code & 0xF);
            else *cb = (uint8_t)(*cb | ((o.code & 0xF) << 4));
          }
        }
      }
    } else {
      for (int64_t k = 0; k < K; ++k) {
        const float s = scale[scale_index(sp, b, r, k, rows, K)];
        orc_elem o = quant_elem(sp->fmt, sp->qmin, sp->qmax, orc_bf16_value(xr[k]), s);
        yr[k] = dequant(o.q, s);
        if (!codes) continue;
        if (sp->fmt == ORC_INT4) {
          uint8_t nib = (uint8_t)(o.code & 0xF); /* two's complement nibble */
          uint8_t* cb = codes + (br * K + k) / 2;
          if ((k & 1) == 0) *cb = nib;
          else *cb = (uint8_t)(*cb | (nib << 4));
        } else {
          codes[br * K + k] = (uint8_t)(o.code & 0xFF);
        }
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Scale gradient (straight-through estimator, LSQ form)                       */
/*   x_hat = s * Q(x / s);  d x_hat / d s = Q(v) - v inside the grid,          */
/*   Q(v) (the clamp bound) where the clamp is active;  d x_hat / d x = 1      */
/*   inside, 0 where clamped.                                                 */
/* ------------------------------------------------------------------------- */

int orc_scale_grad(const orc_spec* sp, const uint16_t* x, const uint16_t* dy, int64_t batch,
                   int64_t rows, int64_t K, const float* scale, const float* tensor_scale,
                   double* dscale, double* dscale_abs, double* dtensor_scale,
                   double* dtensor_scale_abs, uint16_t* dx) {
  if (!spec_ok(sp, K) || batch < 0 || rows < 0 || !x || !dy) return 1;
  const int nvfp4 = sp->fmt == ORC_NVFP4;
  const int dynamic = nvfp4 && sp->mode == ORC_SCALE_DYNAMIC_BLOCK;
  if (nvfp4 && !tensor_scale) return 1;
  if (!dynamic && !scale) return 1;
  const int64_t nrow = batch * rows;
  /* Units that span several rows (per-tensor, per-head, the NVFP4 tensor
   * scale) are summed per row first, then over rows in row order. */
  const int cross_row = dynamic || sp->gran == ORC_PER_TENSOR || sp->gran == ORC_PER_HEAD;
  double* rowsum = NULL;
  double* rowabs = NULL;
  if (cross_row && nrow > 0) {
    rowsum = (double*)calloc((size_t)nrow, sizeof(double));
    rowabs = (double*)calloc((size_t)nrow, sizeof(double));
    if (!rowsum || !rowabs) {
      free(rowsum);
      free(rowabs);
      return 2;
    }
  }
  if (!cross_row) {
    int64_t nunit = (sp->gran == ORC_PER_CHANNEL) ? nrow : nrow * (K / sp->group);
    if (dscale) memset(dscale, 0, (size_t)nunit * sizeof(double));
    if (dscale_abs) memset(dscale_abs, 0, (size_t)nunit * sizeof(double));
  }
#pragma omp parallel for schedule(static)
  for (int64_t br = 0; br < nrow; ++br) {
    const int64_t b = br / rows, r = br % rows;
    const uint16_t* xr = x + br * K;
    const uint16_t* dyr = dy + br * K;
    if (nvfp4) {
      const float g = tensor_scale[b];
      for (int64_t k0 = 0; k0 < K; k0 += 16) {
        const int64_t blk = br * (K / 16) + k0 / 16;
        float sb;
        if (dynamic) {
          double amax = 0.0;
          for (int i = 0; i < 16; ++i) {
            double a = fabs((double)orc_bf16_value(xr[k0 + i]));
            if (a > amax) amax = a;
          }
          sb = fl32(amax / 6.0);
        } else {
          sb = scale[blk];
        }
        int ecode;
        const float sh = nvfp4_block_scale(sb, g, &ecode);
        double bsum = 0.0, babs = 0.0;
        for (int i = 0; i < 16; ++i) {
          orc_elem o = quant_elem(ORC_NVFP4, 0, 0, orc_bf16_value(xr[k0 + i]), sh);
          double d = (double)orc_bf16_value(dyr[k0 + i]);
          double term = o.clipped ? o.q : (o.q - (double)o.v);
          bsum += d * term;
          babs += fabs(d * term);
          if (dx) dx[br * K + k0 + i] = o.clipped ? (uint16_t)0 : dyr[k0 + i];
        }
        if (dynamic) {
          /* block code held fixed: d S_hat / d g = dec(code) */
          double dec = orc_e4m3_decode(ecode);
          rowsum[br] += dec * bsum;
          rowabs[br] += fabs(dec) * babs;
        } else {
          /* straight-through E4M3 rounding of the block scale: d S_hat / d S_b = 1 */
          if (dscale) dscale[blk] = bsum;
          if (dscale_abs) dscale_abs[blk] = babs;
        }
      }
    } else {
      for (int64_t k = 0; k < K; ++k) {
        const int64_t u = scale_index(sp, b, r, k, rows, K);
        const float s = scale[u];
        orc_elem o = quant_elem(sp->fmt, sp->qmin, sp->qmax, orc_bf16_value(xr[k]), s);
        double d = (double)orc_bf16_value(dyr[k]);
        double term = o.clipped ? o.q : (o.q - (double)o.v);
        double t = d * term;
        if (cross_row) {
          rowsum[br] += t;
          rowabs[br] += fabs(t);
        } else {
          if (dscale) dscale[u] += t;
          if (dscale_abs) dscale_abs[u] += fabs(t);
        }
        if (dx) dx[br * K + k] = o.clipped ? (uint16_t)0 : dyr[k];
      }
    }
  }
  if (cross_row) {
    if (dynamic) {
      for (int64_t b = 0; b < batch; ++b) {
        double s = 0.0, a = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
          s += rowsum[b * rows + r];
          a += rowabs[b * rows + r];
        }
        if (dtensor_scale) dtensor_scale[b] = s;
        if (dtensor_scale_abs) dtensor_scale_abs[b] = a;
      }
    } else if (sp->gran == ORC_PER_TENSOR) {
      for (int64_t b = 0; b < batch; ++b) {
        double s = 0.0, a = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
          s += rowsum[b * rows + r];
          a += rowabs[b * rows + r];
        }
        if (dscale) dscale[b] = s;
        if (dscale_abs) dscale_abs[b] = a;
      }
    } else { /* per head: sum over batch for each row index */
      for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0, a = 0.0;
        for (int64_t b = 0; b < batch; ++b) {
          s += rowsum[b * rows + r];
          a += rowabs[b * rows + r];
        }
        if (dscale) dscale[r] = s;
        if (dscale_abs) dscale_abs[r] = a;
      }
    }
  }
  free(rowsum);
  free(rowabs);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Per-head min/max observer and its scale                                     */
/* ------------------------------------------------------------------------- */

/* a < b in the IEEE-754-2019 minimum/maximum order (-0 below +0). */
static int before(float a, float b) {
  if (a == b) return signbit(a) && !signbit(b);
  return a < b;
}

int orc_observer_minmax(const uint16_t* x, int64_t T, int64_t H, int64_t D, float* mn, float* mx,
                        int accumulate) {
  if (!x || !mn || !mx || T < 0 || H < 0 || D < 0) return 1;
#pragma omp parallel for schedule(static)
  for (int64_t h = 0; h < H; ++h) {
    float lo = accumulate ? mn[h] : INFINITY;
    float hi = accumulate ? mx[h] : -INFINITY;
    for (int64_t t = 0; t < T; ++t) {
      const uint16_t* row = x + (t * H + h) * D;
      for (int64_t d = 0; d < D; ++d) {
        float v = orc_bf16_value(row[d]);
        if (before(v, lo)) lo = v;
        if (before(hi, v)) hi = v;
      }
    }
    mn[h] = lo;
    mx[h] = hi;
  }
  return 0;
}

int orc_minmax_scale(const float* mn, const float* mx, int64_t H, double qmax, float* scale) {
  if (!mn || !mx || !scale || H < 0 || !(qmax > 0)) return 1;
  for (int64_t h = 0; h < H; ++h) {
    double a = fabs((double)mn[h]), b = fabs((double)mx[h]);
    double amax = a > b ? a : b;
    scale[h] = fl32(amax / qmax);
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Scale initialisation from the data (amax / qmax)                           */
/* ------------------------------------------------------------------------- */

int orc_scale_init(const orc_spec* sp, const uint16_t* x, int64_t batch, int64_t rows, int64_t K,
                   float* scale, float* tensor_scale) {
  if (!spec_ok(sp, K) || batch < 0 || rows < 0 || !x) return 1;
  const int nvfp4 = sp->fmt == ORC_NVFP4;
  const int dynamic = nvfp4 && sp->mode == ORC_SCALE_DYNAMIC_BLOCK;
  if (nvfp4 && !tensor_scale) return 1;
  if (!dynamic && !scale) return 1;
  const int64_t nrow = batch * rows;
  if (nvfp4) {
    for (int64_t b = 0; b < batch; ++b) {
      double amax = 0.0;
      for (int64_t i = 0; i < rows * K; ++i) {
        double a = fabs((double)orc_bf16_value(x[b * rows * K + i]));
        if (a > amax) amax = a;
      }
      tensor_scale[b] = fl32(amax / (448.0 * 6.0));
    }
    if (dynamic) return 0;
#pragma omp parallel for schedule(static)
    for (int64_t blk = 0; blk < nrow * (K / 16); ++blk) {
      double amax = 0.0;
      for (int i = 0; i < 16; ++i) {
        double a = fabs((double)orc_bf16_value(x[blk * 16 + i]));
        if (a > amax) amax = a;
      }
      scale[blk] = fl32(amax / 6.0);
    }
    return 0;
  }
  const double qmax = (sp->fmt == ORC_FP8_E4M3) ? 448.0 : (double)sp->qmax;
  int64_t nunit;
  switch (sp->gran) {
    case ORC_PER_TENSOR: nunit = batch; break;
    case ORC_PER_CHANNEL: nunit = nrow; break;
    case ORC_PER_GROUP: nunit = nrow * (K / sp->group); break;
    default: nunit = rows; break;
  }
  double* amax = (double*)calloc((size_t)(nunit > 0 ? nunit : 1), sizeof(double));
  if (!amax) return 2;
  for (int64_t br = 0; br < nrow; ++br) {
    const int64_t b = br / rows, r = br % rows;
    for (int64_t k = 0; k < K; ++k) {
      double a = fabs((double)orc_bf16_value(x[br * K + k]));
      int64_t u = scale_index(sp, b, r, k, rows, K);
      if (a > amax[u]) amax[u] = a;
    }
  }
  for (int64_t u = 0; u < nunit; ++u) scale[u] = fl32(amax[u] / qmax);
  free(amax);
  return 0;
}
