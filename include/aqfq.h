/*
 * aqfq.h -- C ABI of libaqfq: learnable-scale fake-quant (quantize-dequantize)
 * of frozen BF16 weights and activations on one NVIDIA GB300 (sm_103a).
 *
 * What the calls compute (the method, restated from the pages):
 *   - AngelSlim mcore_qad article, section 1: weights stay frozen in BF16; in
 *     the forward pass weights and activations are quantized then dequantized
 *     (fake-quant); the quantizer scales are the only trainable tensors.
 *   - Same article, section 2.3: weight fake-quant is applied transparently to
 *     module.weight, activations are fake-quantized before the matmul, the
 *     gradient flows to the scales; router and output layer are not quantized
 *     (callers simply do not pass them here).
 *   - Same article, section 2.4: each MoE layer's experts become one 3D stack
 *     [E, N, K] that is fake-quantized in one vectorised pass.
 *   - Same article, section 3: formats nvfp4, nvfp4a16, w4a16 (INT4), w8a8
 *     (INT8), fp8; section 6: scale sources learnable / dynamic / calibrated.
 *   - "QAT + DeepSpeed ZeRO-3" (AngelSlim docs), "Quantizer changes": the
 *     fake-quant output is cast back to the input dtype (BF16 in, BF16 out);
 *     "Quantizer initial values": a PTQ weight scale is about max|W|/448.
 *   - msModelSlim "multi-card quantization adaptation guide", "FA3Quant"
 *     steps 3-4: per-head min/max observer with a running merge; qparams are
 *     computed from the merged min/max.
 *
 * Arithmetic (identical for every format; all binary32, round to nearest even):
 *   v     = x / s                (IEEE division; s = 0 gives v = +-0, sign of x)
 *   q     = grid(v)              nearest grid value, ties to the even code,
 *                                saturating at the grid's ends
 *   x_hat = bf16(q * s)          product rounded to binary32, then to BF16
 *   grid: INT8/INT4 integers in [qmin, qmax] (integer 0 has no sign);
 *         FP8 E4M3 (largest 448); NVFP4 E2M1 (largest 6), sign of zero kept.
 *   NVFP4 block scale: e_b = E4M3(S_b / g) (saturating), s = dec(e_b) * g.
 *   Scale gradient (straight-through estimator, LSQ form):
 *         d x_hat / d s = q - v if the clamp is inactive, q if it is active
 *         (INT: v <= qmin or v >= qmax; FP: |v| >= largest finite value);
 *         d x_hat / d x = 1 if inactive, 0 if active.
 *
 * Rows of K = 8 * odd elements (K % 8 == 0 but K % 16 != 0) are accepted for
 * per-tensor, per-channel and per-head INT8 / INT4 / FP8 (8-element chunks);
 * NVFP4 and per-group specs need K % 16 == 0 (their blocks and groups are 16
 * elements or more).
 *
 * Layouts (all row-major, K contiguous, BF16 as 16-bit patterns):
 *   x, y, dy, dx : [batch, rows, K]   (batch = experts E for stacks, else 1;
 *                                      [T, H, D] for per-head activations)
 *   scale        : AQFQ_PER_TENSOR [batch]; AQFQ_PER_CHANNEL [batch, rows];
 *                  AQFQ_PER_GROUP [batch, rows, K/group]; AQFQ_PER_HEAD [rows]
 *                  (shared by all batch entries); NVFP4 learned [batch, rows, K/16]
 *   tensor_scale : NVFP4 only, [batch] float
 *   codes        : optional; INT8 / FP8: one byte per element [batch, rows, K];
 *                  INT4 / NVFP4: two per byte [batch, rows, K/2], element k even
 *                  in the low nibble (INT4 nibbles are two's complement,
 *                  E2M1 nibbles are sign<<3 | exponent<<1 | mantissa)
 *   block_codes  : optional, NVFP4 only: E4M3 byte per block [batch, rows, K/16]
 *
 * Ownership and errors: every pointer is device memory owned by the caller;
 * the library allocates nothing and keeps no state between calls (it caches
 * the SM count of each device).  Calls are asynchronous on `stream` (a
 * cudaStream_t passed as void*, NULL = legacy default stream) and never
 * synchronise.  Arguments are checked on the host before anything is
 * launched; a rejected call launches nothing and returns a status:
 *   AQFQ_ERR_NULL         a required pointer is NULL (a buffer with no
 *                         elements may be NULL)
 *   AQFQ_ERR_SHAPE        negative size, K % 8 != 0, K % 16 != 0 for NVFP4
 *                         or any per-group spec (K % group != 0), or a size
 *                         beyond the limits stated per call
 *   AQFQ_ERR_ALIGN        x / y / dy / dx not 16-byte aligned (32-byte aligned
 *                         tensors take 256-bit accesses, 16-byte aligned ones
 *                         128-bit accesses; the results are the same); codes
 *                         not aligned to one chunk's codes: 16 bytes (INT8 /
 *                         FP8) or 8 bytes (INT4 / NVFP4) when K % 16 == 0,
 *                         8 or 4 bytes when K = 8 * odd; float arrays not
 *                         4-byte aligned; workspace not 8-byte
 *   AQFQ_ERR_UNSUPPORTED  a format / granularity / mode combination the
 *                         library does not implement
 *   AQFQ_ERR_WORKSPACE    workspace smaller than aqfq_scale_grad_workspace_bytes
 *   AQFQ_ERR_CUDA         a launch failed (cudaGetLastError after launching)
 * Inputs are assumed finite (no NaN / Inf); the library does not check them.
 */
#ifndef AQFQ_H
#define AQFQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum aqfq_status {
  AQFQ_OK = 0,
  AQFQ_ERR_NULL = 1,
  AQFQ_ERR_SHAPE = 2,
  AQFQ_ERR_ALIGN = 3,
  AQFQ_ERR_UNSUPPORTED = 4,
  AQFQ_ERR_WORKSPACE = 5,
  AQFQ_ERR_CUDA = 6
} aqfq_status;

/* element formats (AngelSlim mcore_qad article, section 3) */
enum { AQFQ_INT8 = 0, AQFQ_INT4 = 1, AQFQ_FP8_E4M3 = 2, AQFQ_NVFP4 = 3 };
/* scale granularities */
enum { AQFQ_PER_TENSOR = 0, AQFQ_PER_CHANNEL = 1, AQFQ_PER_GROUP = 2, AQFQ_PER_HEAD = 3 };
/* scale sources (same article, section 6: learnable / dynamic) */
enum { AQFQ_SCALE_LEARNED = 0, AQFQ_SCALE_DYNAMIC_BLOCK = 1 };

/* Quantizer description.
 *   fmt   : AQFQ_INT8 | AQFQ_INT4 | AQFQ_FP8_E4M3 | AQFQ_NVFP4
 *   gran  : AQFQ_PER_*; NVFP4 requires AQFQ_PER_GROUP with group 16
 *   group : elements per scale along K for AQFQ_PER_GROUP: a power of two in
 *           [16, 512] (128 for w4a16 INT4), ignored otherwise
 *   qmin, qmax : integer grid for INT8 (within [-128, 127]) and INT4 (within
 *           [-8, 7]), qmin < 0 < qmax; ignored for FP8 / NVFP4
 *   mode  : AQFQ_SCALE_LEARNED (scale given by the caller), or, NVFP4 only,
 *           AQFQ_SCALE_DYNAMIC_BLOCK: block scale S_b = amax_b / 6 computed
 *           from the data, the tensor scale g is the learned one. */
typedef struct aqfq_qspec {
  int32_t fmt;
  int32_t gran;
  int32_t group;
  int32_t qmin;
  int32_t qmax;
  int32_t mode;
} aqfq_qspec;

/* Fake-quant forward: y = x_hat (BF16, same shape as x) and, if non-NULL, the
 * packed codes and (NVFP4) the E4M3 block codes.
 * Source: AngelSlim mcore_qad article, sections 1 and 2.3 (weights and
 * activations quantized-dequantized in the forward), section 3 (formats);
 * "QAT + DeepSpeed ZeRO-3", "Quantizer changes" (output cast back to BF16).
 *   x            device, [batch, rows, K] BF16
 *   scale        device, shaped by spec->gran (NULL only for NVFP4 dynamic)
 *   tensor_scale device, [batch] float (NVFP4), else ignored
 *   y            device, [batch, rows, K] BF16; must not overlap x.  May be
 *                NULL when codes are requested: real-quant export, which
 *                writes only the packed codes (and block codes).
 * Export layouts (the codes are the deployment tensors, byte for byte):
 *   INT4 (w4a16): codes viewed as int32 [batch, rows, K/8] hold element 8j+i
 *     in bits 4i..4i+3 (pack-quantized order), scale per group as given;
 *   FP8: codes are float8_e4m3fn [batch, rows, K] with the per-channel /
 *     per-tensor float32 scale;
 *   NVFP4: codes uint8 [batch, rows, K/2] (element 2j in the low nibble),
 *     block_codes float8_e4m3fn [batch, rows, K/16], dequantised value
 *     e2m1 * e4m3 * tensor_scale (a "global scale" stored as its reciprocal
 *     by some deployment formats is 1 / tensor_scale).
 * (AngelSlim mcore_qad article, section 3: format names map 1:1 to the
 * deployment side's layouts; "QAT + DeepSpeed ZeRO-3": save_format=real.)
 * Limits: rows * K / 16 < 2^32 per batch entry (rows * K / 8 when K % 16 != 0). */
aqfq_status aqfq_qdq_fwd(const aqfq_qspec* spec, const void* x, int64_t batch, int64_t rows,
                         int64_t K, const float* scale, const float* tensor_scale, void* y,
                         uint8_t* codes, uint8_t* block_codes, void* stream);

/* The same forward over a 3D stack of MoE expert weights w [E, N, K]: one
 * vectorised pass over every expert, per-expert tensor scale (NVFP4).
 * Source: AngelSlim mcore_qad article, section 2.4 (3D stacked expert
 * weights, whole-stack vectorised fake-quant, then one grouped GEMM).
 * Arguments as aqfq_qdq_fwd with batch = E, rows = N. */
aqfq_status aqfq_grouped_qdq(const aqfq_qspec* spec, const void* w, int64_t E, int64_t N,
                             int64_t K, const float* scale, const float* tensor_scale, void* y,
                             uint8_t* codes, uint8_t* block_codes, void* stream);

/* Straight-through scale gradient: dscale = sum over each scale's unit of
 * dy * (d x_hat / d s); optional STE input gradient dx = dy where the clamp
 * is inactive, +0 where active.  Weights are frozen, so callers pass dx =
 * NULL for weights.
 * Source: AngelSlim mcore_qad article, section 1 (only the scales are
 * optimised) and 2.3 (the gradient flows to the scale through the fake-quant).
 *   dy            device, [batch, rows, K] BF16, upstream gradient dL/dx_hat
 *   dscale        device, shaped like scale; learned modes only (NULL for
 *                 NVFP4 dynamic)
 *   dtensor_scale device, [batch] float: NVFP4 dynamic mode only (gradient of
 *                 the learned tensor scale with the block codes held fixed);
 *                 must be NULL otherwise
 *   dx            device, optional, [batch, rows, K] BF16
 *   accumulate    0: overwrite dscale / dtensor_scale; else add to them
 *   workspace     device scratch, >= aqfq_scale_grad_workspace_bytes(...)
 *                 bytes (0 bytes for per-channel / per-group / NVFP4 learned;
 *                 per-tensor, per-head and the NVFP4 tensor scale need it; the
 *                 result is deterministic: fixed reduction order).  Per-tensor
 *                 and tensor-scale reductions keep a counter in its first 16
 *                 bytes, which the call zeroes on the stream itself: the
 *                 contents need no initialisation.
 * Per-head (x [T, H, D], scale [H], learnable per-head activation scale, e.g.
 * FP8 attention / KV activations; msModelSlim guide, "FA3Quant"): requires
 * H * D / 16 <= 2^24 (H * D / 8 when D % 16 != 0). */
aqfq_status aqfq_scale_grad(const aqfq_qspec* spec, const void* x, const void* dy, int64_t batch,
                            int64_t rows, int64_t K, const float* scale,
                            const float* tensor_scale, float* dscale, float* dtensor_scale,
                            void* dx, int accumulate, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Forward and scale gradient in one pass: y = x_hat exactly as aqfq_qdq_fwd
 * writes it (no codes) and dscale / dtensor_scale / dx exactly as
 * aqfq_scale_grad writes them, from one read of x and dy.  For callers that
 * hold the upstream gradient when they need the forward's output: the
 * fake-quant forward recomputed in the backward pass (activation
 * checkpointing), where the weight gradient dW, the fake-quant's upstream
 * gradient, is formed without x_hat while x_hat is needed for the input
 * gradient.  x is read once instead of twice and one launch replaces two.
 * Source: AngelSlim mcore_qad article, sections 1 and 2.3 (forward
 * fake-quant; the gradient flows to the scale through it).
 * Arguments as aqfq_scale_grad, plus
 *   y            device, [batch, rows, K] BF16, required; must not overlap x,
 *                dy or dx
 * The workspace is the one aqfq_scale_grad_workspace_bytes gives. */
aqfq_status aqfq_qdq_fwd_grad(const aqfq_qspec* spec, const void* x, const void* dy,
                              int64_t batch, int64_t rows, int64_t K, const float* scale,
                              const float* tensor_scale, void* y, float* dscale,
                              float* dtensor_scale, void* dx, int accumulate, void* workspace,
                              size_t workspace_bytes, void* stream);

/* aqfq_scale_grad for callers that cannot allocate device memory (no
 * counterpart in the pages: a library convenience).  Some callers cannot hand
 * over a scratch buffer: a plugin inside a framework that owns all device
 * memory through its own pool and gives the plugin no allocation hook, or a
 * latency-critical path where a cudaMalloc, which may synchronise the device,
 * is not acceptable.  This call takes the scratch of the per-tensor, NVFP4
 * tensor-scale and per-head reductions from a 128 KiB array inside the
 * library (held by every GPU that loads the library until the process exits)
 * and allocates nothing.  Arguments and results as aqfq_scale_grad without
 * the workspace.
 *   - Returns AQFQ_ERR_WORKSPACE when aqfq_scale_grad_workspace_bytes(...)
 *     exceeds 128 KiB (a 16-byte counter and 16382 partial sums).  Per-tensor
 *     and tensor-scale gradients fit for up to about 16380 batch entries;
 *     per-head gradients (x [T, H, D]) fit only while T * H * D / 16 <= 16384.
 *   - All calls share the array: calls whose kernels may overlap on the GPU
 *     (unordered streams) race.  Nothing needs clearing between calls.
 *   - The array's device address is looked up for the device current at the
 *     call, once per device and CUDA context (cached under the context's
 *     unique ID, so a device reset leads to a fresh lookup).  The first call
 *     on a device may load the library's device code there: make it before
 *     any stream capture. */
aqfq_status aqfq_scale_grad_noalloc(const aqfq_qspec* spec, const void* x, const void* dy,
                                    int64_t batch, int64_t rows, int64_t K, const float* scale,
                                    const float* tensor_scale, float* dscale,
                                    float* dtensor_scale, void* dx, int accumulate,
                                    void* stream);

/* Bytes of device scratch aqfq_scale_grad needs for these arguments (0 when
 * none); returns 0 for arguments aqfq_scale_grad would reject. */
size_t aqfq_scale_grad_workspace_bytes(const aqfq_qspec* spec, int64_t batch, int64_t rows,
                                       int64_t K);

/* Per-head min/max observer over x [T, H, D] (BF16): min_out[h] / max_out[h]
 * = min / max of x[:, h, :] (exact BF16 values as float; -0 orders below +0).
 * accumulate != 0 merges with the values already in min_out / max_out (the
 * running min/max of successive calibration batches; merging shards this way
 * equals one pass over all of them).  With T = 0 and accumulate = 0 the
 * result is +inf / -inf.
 * Source: msModelSlim guide, "FA3Quant" steps 3-4 (per-head local min/max,
 * min-of-mins / max-of-maxes merge).
 * Limits: D % 8 == 0; H * D / 16 <= 2^24 (H * D / 8 when D % 16 != 0); x
 * 16-byte aligned. */
aqfq_status aqfq_observer_minmax(const void* x, int64_t T, int64_t H, int64_t D, float* min_out,
                                 float* max_out, int accumulate, void* stream);

/* Per-head symmetric scale from the observer: scale[h] = max(|min|, |max|) /
 * qmax (binary32 division; qmax = 448 for E4M3).  The result feeds
 * aqfq_qdq_fwd with gran = AQFQ_PER_HEAD.
 * Source: msModelSlim guide, "FA3Quant" step 3 (qparams from the merged
 * min/max); "QAT + DeepSpeed ZeRO-3", "Quantizer initial values" (amax/448). */
aqfq_status aqfq_minmax_scale(const float* min_in, const float* max_in, int64_t H, float qmax,
                              float* scale_out, void* stream);

/* Scale initialisation from the data: every scale = amax over its unit /
 * qmax (INT: spec->qmax; FP8: 448).  NVFP4 learned: scale = amax_b / 6 per
 * 16-element block and tensor_scale[b] = amax / (448 * 6) per batch entry;
 * NVFP4 dynamic: tensor_scale only (scale may be NULL).
 * Source: "QAT + DeepSpeed ZeRO-3", "Quantizer initial values" (PTQ scale
 * about max|W| / 448); the INT8 rule amax / 127 is the same rule on the
 * integer grid. */
aqfq_status aqfq_scale_init(const aqfq_qspec* spec, const void* x, int64_t batch, int64_t rows,
                            int64_t K, float* scale, float* tensor_scale, void* stream);

/* Fused NVFP4 weight fake-quant + grouped GEMM (nvfp4a16: NVFP4 weights, BF16
 * activations).  For each expert e and each row m of x with
 * m_offsets[e] <= m < m_offsets[e+1]:
 *     y[m, n] = sum_k x[m, k] * w_hat_e[n, k]
 * where w_hat_e is the NVFP4 fake-quant of w[e] with learned block scales and
 * the expert's tensor scale, bit for bit as aqfq_grouped_qdq computes it; the
 * fake-quantized weight is formed in shared memory and never written to
 * device memory.  Products accumulate in FP32 on the tensor cores (tcgen05);
 * y is rounded to BF16.
 * Source: AngelSlim mcore_qad article, section 2.4 (vectorised fake-quant of
 * the whole expert stack, then one grouped GEMM for every expert) and section
 * 3 (format nvfp4a16).
 *   x            device, [total_m, K] BF16, rows grouped by expert
 *   m_offsets    device int32 [E + 1]: 0 = m_offsets[0] <= ... <= m_offsets[E]
 *                = total_m (the kernel clamps them to [0, total_m])
 *   w            device, [E, N, K] BF16;  scale [E, N, K/16] f32;
 *   tensor_scale [E] f32;  y  device, [total_m, N] BF16
 *   error_flag   optional device int32, set to 1 if a pipeline wait of the
 *                kernel timed out (y is then incomplete); never cleared
 * Limits: N % 128 == 0, K % 64 == 0, K > 0, (total_m + 511) / 512 + E <= 65535;
 * x, w, y 32-byte aligned.  Allocates nothing; asynchronous on `stream`. */
aqfq_status aqfq_grouped_qdq_gemm(const void* x, const int32_t* m_offsets, int64_t total_m,
                                  const void* w, const float* scale, const float* tensor_scale,
                                  int64_t E, int64_t N, int64_t K, void* y, int32_t* error_flag,
                                  void* stream);

/* ---- distillation losses (QAD: the student is the fake-quantized model) ----
 * Loss between student and teacher logits with the gradient for the student
 * logits, without any [tokens, vocab] intermediate.
 * Sources: AngelSlim "QAT + DeepSpeed ZeRO-3" page, table "KD variants
 * (loss_type)" (kl = KL(teacher || student), rkl = KL(student || teacher),
 * mse, cakld = conf * rkl + (1 - conf) * fkl with conf the teacher's
 * probability of the label, the temperature form T^2 * KL, kl_top_K /
 * r_kl_top_K) and its cakld formula (per position, only where the label is
 * not -100, then the mean); AngelSlim mcore_qad article, section 2.5
 * (distill_topk: KL on the teacher's top-k tokens only).
 * Per position with a label in [0, V), a = teacher / tau, b = student / tau,
 * U = every token (topk = 0) or the teacher's topk largest logits (equal
 * values lower index first; -0 equals +0), p_t = softmax over U of a,
 * p_s = softmax over U of b:
 *   fkl = tau^2 sum_U p_t (log p_t - log p_s)   rkl = tau^2 sum_U p_s (log p_s - log p_t)
 *   conf = softmax(a)[label] over the whole vocabulary
 *   loss = fkl (AQFQ_KD_KL) | rkl (AQFQ_KD_RKL) | conf rkl + (1 - conf) fkl
 *          (AQFQ_KD_CAKLD) | mean over the vocabulary of (s - t)^2 (AQFQ_KD_MSE)
 * Positions whose label lies outside [0, V) (the ignore index -100 among them)
 * carry no loss and no gradient.  losses[0..2] = the means over the valid
 * positions of (loss, fkl, rkl) (0 when there is none).
 *   student, teacher device [T, V] BF16, V contiguous, 16-byte aligned
 *   labels           device int32 [T]
 *   topk             0 = whole vocabulary, else 1 <= topk <= V
 *   temperature      tau > 0 (1 = plain); AQFQ_KD_MSE needs tau = 1, topk = 0
 *   grad_scale       the gradient written is grad_scale * d losses[0] / d student
 *   losses           device float [3], written
 *   token_loss       optional device float [T]: loss per position (0 if ignored)
 *   dstudent         optional device [T, V] BF16: the gradient (zeros outside
 *                    the support and at ignored positions)
 *   topk_idx         optional device int32 [T, topk] (topk > 0 only): the
 *                    support in ascending vocabulary order, -1 rows at ignored
 *                    positions
 *   workspace        device, aqfq_kd_workspace_bytes(T) bytes, 16-byte aligned
 * Limits: V % 8 == 0, 8 <= V, V up to the shared-memory bound (about 400k on
 * GB300: each of 8 CTAs holds 1/8 of both rows).  Arithmetic in binary32 with
 * hardware base-2 exponentials; the tests state the error bound.
 * Launches three kernels (count, loss, mean); asynchronous on `stream`. */
typedef enum aqfq_kd_type {
  AQFQ_KD_KL = 0,
  AQFQ_KD_RKL = 1,
  AQFQ_KD_CAKLD = 2,
  AQFQ_KD_MSE = 3
} aqfq_kd_type;

size_t aqfq_kd_workspace_bytes(int64_t T);

aqfq_status aqfq_kd_loss(int kd_type, const void* student, const void* teacher,
                         const int32_t* labels, int64_t T, int64_t V, int32_t topk,
                         float temperature, float grad_scale, float* losses, float* token_loss,
                         void* dstudent, int32_t* topk_idx, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Diagnostic (the pages have no counterpart): checks the bounded-wait path
 * that the GEMM's pipeline uses when a stage never arrives.  One thread waits
 * on an mbarrier phase that nothing completes, polling at most `polls` times
 * (1 <= polls <= 2^22, backing off to 256 ns per poll), then sets *flag = 1
 * (device int32, 4-byte aligned) and returns; the context stays usable.
 * Asynchronous on `stream`; allocates nothing. */
aqfq_status aqfq_selftest_wait_timeout(int32_t* flag, uint32_t polls, void* stream);

/* Diagnostic (the pages have no counterpart): the grid rounding step of the
 * fake-quant kernels applied to binary32 values given directly.  codes[i] is
 * the code that the forward and gradient kernels give a quotient v[i]: INT8 /
 * INT4 two's-complement codes of round-half-even(clamp(v, qmin, qmax)) (one
 * byte per value; INT4 in the low nibble), E4M3 (spec->fmt = AQFQ_FP8_E4M3)
 * bytes and E2M1 (AQFQ_NVFP4) nibbles of the saturating round-to-nearest-even
 * conversion of |v| with the sign of v as the code's sign bit.  Lets a test
 * compare that step with the oracle for every binary32 value.
 *   spec   fmt and (INT) qmin / qmax as for the fake-quant calls
 *   v      device float [n], 4-byte aligned;  codes  device uint8 [n]
 * Asynchronous on `stream`; allocates nothing. */
aqfq_status aqfq_selftest_grid_codes(const aqfq_qspec* spec, const float* v, int64_t n,
                                     uint8_t* codes, void* stream);

/* Static text for a status code. */
const char* aqfq_status_string(aqfq_status status);

/* ABI version (major * 100 + minor). */
int aqfq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* AQFQ_H */
