/*
 * aqfq_oracle.h -- plain, slow CPU oracle for learnable-scale fake-quant.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link or
 * load this library: only the test suite, the smoke check and the CPU baseline
 * leg of the benchmark use it.  It shares no source with the CUDA library.
 *
 * What it computes (the method, restated from the pages):
 *   - AngelSlim mcore_qad article, section 1 ("why training only the scale is
 *     enough"): weights stay frozen in BF16; the forward quantizes and then
 *     dequantizes weights and activations; the scales are the only trainable
 *     tensors.
 *   - Same article, section 3: the formats nvfp4, w4a16 (INT4), w8a8 (INT8),
 *     fp8.  Section 2.4: the experts of one MoE layer are one 3D stack that is
 *     fake-quantized in one vectorised pass.
 *   - "QAT + DeepSpeed ZeRO-3" (AngelSlim docs), "Quantizer changes": the
 *     fake-quant output is cast back to the input dtype (BF16 here).
 *     "Quantizer initial values": a PTQ weight scale is about max|W|/448.
 *   - msModelSlim "multi-card quantization adaptation guide", "FA3Quant"
 *     steps 3-4: per-head min/max observer, running min/max merge, qparams
 *     computed from the merged min/max.
 *
 * Arithmetic: every floating-point step is done in double; where the method
 * rounds to binary32 (the quotient v = x/s, the product q*s, block scales)
 * the double result is rounded to float, which for one division or one
 * product of floats gives the correctly rounded binary32 value.  Grid
 * rounding (INT, E4M3, E2M1) is the nearest grid value, ties to the even
 * code, saturating at the largest finite value, sign of zero kept.
 *
 * Layout conventions (same meaning as the CUDA library, written separately):
 *   x, dy, y, dx : [batch, rows, K] BF16 bit patterns (uint16), K contiguous.
 *   scale        : PER_TENSOR [batch]; PER_CHANNEL [batch, rows];
 *                  PER_GROUP [batch, rows, K/group]; PER_HEAD [rows].
 *   tensor_scale : NVFP4 only, [batch] float.
 *   codes        : INT8 / FP8 one byte per element; INT4 / NVFP4 two per byte,
 *                  element k even in the low nibble.
 *   block_codes  : NVFP4 only, E4M3 byte per 16-element block [batch, rows, K/16].
 */
#ifndef AQFQ_ORACLE_H
#define AQFQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_INT8 = 0, ORC_INT4 = 1, ORC_FP8_E4M3 = 2, ORC_NVFP4 = 3 };
enum { ORC_PER_TENSOR = 0, ORC_PER_CHANNEL = 1, ORC_PER_GROUP = 2, ORC_PER_HEAD = 3 };
enum { ORC_SCALE_LEARNED = 0, ORC_SCALE_DYNAMIC_BLOCK = 1 };

typedef struct {
  int32_t fmt, gran, group, qmin, qmax, mode;
} orc_spec;

/* ---- format primitives (exposed so the tests can pin them) ---- */
double   orc_e4m3_decode(int code);          /* NaN for 0x7F / 0xFF */
double   orc_e2m1_decode(int code);
int      orc_e4m3_encode(double v);          /* nearest finite, ties even, satfinite */
int      orc_e2m1_encode(double v);
double   orc_int_round(double v, int qmin, int qmax);
uint16_t orc_bf16_round(float f);            /* binary32 -> bf16 bits, nearest even */
float    orc_bf16_value(uint16_t bits);
float    orc_div32(float a, float b);        /* correctly rounded binary32 a/b */

/* ---- the path ---- */
int orc_qdq_fwd(const orc_spec* sp, const uint16_t* x, int64_t batch, int64_t rows,
                int64_t K, const float* scale, const float* tensor_scale,
                uint16_t* y, uint8_t* codes, uint8_t* block_codes);

/* dscale[u] = sum over the unit of dy * term; dscale_abs[u] = sum of |dy * term|
 * (the second is the condition denominator the tests use).  dtensor_scale /
 * dtensor_scale_abs: NVFP4 dynamic mode, per batch entry.  dx: STE input grad.
 * Any output pointer may be NULL. */
int orc_scale_grad(const orc_spec* sp, const uint16_t* x, const uint16_t* dy, int64_t batch,
                   int64_t rows, int64_t K, const float* scale, const float* tensor_scale,
                   double* dscale, double* dscale_abs, double* dtensor_scale,
                   double* dtensor_scale_abs, uint16_t* dx);

/* x [T,H,D]; mn/mx [H]; accumulate != 0 merges with the values already there. */
int orc_observer_minmax(const uint16_t* x, int64_t T, int64_t H, int64_t D,
                        float* mn, float* mx, int accumulate);
/* scale[h] = fl32(max(|mn[h]|, |mx[h]|) / qmax) */
int orc_minmax_scale(const float* mn, const float* mx, int64_t H, double qmax, float* scale);

/* scale initialisation from the data: amax of each unit / qmax of the format.
 * NVFP4 learned: block scale amax_b/6 and tensor scale amax/(448*6);
 * NVFP4 dynamic: tensor scale only.  scale may be NULL in dynamic mode. */
int orc_scale_init(const orc_spec* sp, const uint16_t* x, int64_t batch, int64_t rows,
                   int64_t K, float* scale, float* tensor_scale);

int orc_num_threads(void);
void orc_set_num_threads(int n);

/* ---- distillation losses (kd_oracle.c) ----
 * kd_type: 0 kl (forward KL), 1 rkl (reverse KL), 2 cakld, 3 mse.
 * student, teacher: [T, V] BF16 bits; labels [T] (outside [0, V) = ignored).
 * topk: 0 = whole vocabulary, else the teacher's top-K support (K <= V).
 * losses[3] = means over valid positions of {loss, tau^2 fkl, tau^2 rkl};
 * tok[T, 3] the same per position; cond[T, 2] error scales (KL family, mse);
 * dstudent / gmag [T, V] (optional): gradient of losses[0] * grad_scale and
 * its error scale; topk_idx [T, K] (optional, topk > 0): the support in
 * ascending vocabulary order, -1 for ignored positions. Returns 0 on success. */
int orc_kd_loss(int kd_type, const uint16_t* student, const uint16_t* teacher,
                const int32_t* labels, int64_t T, int64_t V, int32_t topk, double temperature,
                double grad_scale, double* losses, double* tok, double* cond, double* dstudent,
                double* gmag, int32_t* topk_idx);

#ifdef __cplusplus
}
#endif
#endif
