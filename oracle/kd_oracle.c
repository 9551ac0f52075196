/*
 * kd_oracle.c -- plain, slow CPU oracle for the distillation losses of
 * scale-only QAD (TEST INFRASTRUCTURE ONLY: only the test suite, the smoke
 * check and the CPU baseline leg of the benchmark load it; it shares no code
 * with the CUDA library).
 *
 * What it computes, restated from the pages:
 *   - "QAT + DeepSpeed ZeRO-3" (AngelSlim docs), table "KD variants
 *     (loss_type)": kl = KL(teacher || student) (forward KL), rkl =
 *     KL(student || teacher) (reverse KL), mse = MSE of student and teacher
 *     logits, each averaged over the valid positions; cakld mixes the two KLs
 *     per position with the teacher's probability of the label as the weight,
 *     conf * rkl + (1 - conf) * fkl, only where labels != -100; kd is the
 *     temperature form T^2 * KL of the softened distributions; kl_top_K /
 *     r_kl_top_K take the KL over the teacher's top-K tokens only.
 *   - Same page, the cakld formula block: forward_kl = KL(log_softmax(student),
 *     softmax(teacher)) in the kl_div(input, target) convention, i.e.
 *     sum p_t (log p_t - log p_s); backward_kl the same with the roles swapped;
 *     conf = softmax(teacher) gathered at the label.
 *   - AngelSlim mcore_qad article, section 2.5: with distill_topk > 0 the KL
 *     is computed on the teacher's top-k tokens only, so that no
 *     [tokens, vocab] tensor is materialised.
 *
 * Readings where the pages leave a step open (each stated once, here):
 *   - top-K support: the K largest teacher logits by value; equal values
 *     (+0 and -0 count as equal) are taken lower vocabulary index first; both
 *     distributions are renormalised over that support (softmax of the
 *     gathered logits); conf always uses the full-vocabulary teacher softmax.
 *   - temperature tau: logits divided by tau, every KL multiplied by tau^2
 *     (the kd form); conf uses the same softened teacher; tau = 1 is plain.
 *   - mse: per position the mean over the vocabulary of (s - t)^2; no
 *     temperature, no top-K.
 *   - labels outside [0, V) (the ignore index -100 among them) carry no loss
 *     and no gradient.
 *   - the reported forward / backward KL diagnostics use the same support and
 *     temperature (tau^2 factor included) as the selected loss.
 *   - the gradient is that of losses[0] (the mean over valid positions) with
 *     respect to the student logits, times grad_scale; conf is a teacher
 *     quantity and gets no gradient.
 *
 * Arithmetic: double throughout, log-sum-exp with the maximum subtracted.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "aqfq_oracle.h"

enum { KD_KL = 0, KD_RKL = 1, KD_CAKLD = 2, KD_MSE = 3 };

static double bf16v(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

typedef struct {
  double v;
  int64_t i;
} vi_pair;

/* larger value first; equal values lower index first */
static int by_value_desc(const void* pa, const void* pb) {
  const vi_pair* a = (const vi_pair*)pa;
  const vi_pair* b = (const vi_pair*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->i < b->i) ? -1 : (a->i > b->i);
}

static int by_index(const void* pa, const void* pb) {
  const int64_t a = *(const int64_t*)pa, b = *(const int64_t*)pb;
  return (a > b) - (a < b);
}

/* log sum_i exp(x[idx[i]]) over n entries (idx NULL: the first n) */
static double logsumexp(const double* x, const int64_t* idx, int64_t n) {
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    const double v = x[idx ? idx[j] : j];
    if (v > m) m = v;
  }
  double z = 0.0;
  for (int64_t j = 0; j < n; ++j) z += exp(x[idx ? idx[j] : j] - m);
  return m + log(z);
}

int orc_kd_loss(int kd_type, const uint16_t* student, const uint16_t* teacher,
                const int32_t* labels, int64_t T, int64_t V, int32_t topk, double temperature,
                double grad_scale, double* losses, double* tok, double* cond, double* dstudent,
                double* gmag, int32_t* topk_idx) {
  if (kd_type < KD_KL || kd_type > KD_MSE || T < 0 || V < 1 || topk < 0 || topk > V) return 1;
  if (!(temperature > 0.0)) return 1;
  if (kd_type == KD_MSE && (topk != 0 || temperature != 1.0)) return 1;
  const double tau = temperature;
  const int64_t K = (topk > 0) ? topk : V;

  int64_t n_valid = 0;
  for (int64_t t = 0; t < T; ++t)
    if (labels[t] >= 0 && labels[t] < V) ++n_valid;
  const double gs = n_valid ? grad_scale / (double)n_valid : 0.0;

  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int64_t t = 0; t < T; ++t) {
    const uint16_t* srow = student + t * V;
    const uint16_t* trow = teacher + t * V;
    double* tk = tok + 3 * t;
    const int valid = labels[t] >= 0 && labels[t] < V;
    tk[0] = tk[1] = tk[2] = 0.0;
    cond[2 * t] = cond[2 * t + 1] = 0.0;
    if (dstudent) memset(dstudent + t * V, 0, (size_t)V * sizeof(double));
    if (gmag) memset(gmag + t * V, 0, (size_t)V * sizeof(double));
    if (topk_idx && topk > 0)
      for (int64_t j = 0; j < K; ++j) topk_idx[t * K + j] = -1;
    if (!valid) continue;

    double* a = (double*)malloc((size_t)V * sizeof(double));  /* teacher / tau */
    double* b = (double*)malloc((size_t)V * sizeof(double));  /* student / tau */
    int64_t* sup = (int64_t*)malloc((size_t)K * sizeof(int64_t));
    if (!a || !b || !sup) {
      free(a);
      free(b);
      free(sup);
      fail = 1;
      continue;
    }
    for (int64_t i = 0; i < V; ++i) {
      a[i] = bf16v(trow[i]) / tau;
      b[i] = bf16v(srow[i]) / tau;
    }

    /* the support: every token, or the teacher's K largest logits */
    if (K < V) {
      vi_pair* pr = (vi_pair*)malloc((size_t)V * sizeof(vi_pair));
      if (!pr) {
        free(a);
        free(b);
        free(sup);
        fail = 1;
        continue;
      }
      for (int64_t i = 0; i < V; ++i) {
        pr[i].v = bf16v(trow[i]);  /* -0 == +0 as values */
        pr[i].i = i;
      }
      qsort(pr, (size_t)V, sizeof(vi_pair), by_value_desc);
      for (int64_t j = 0; j < K; ++j) sup[j] = pr[j].i;
      free(pr);
      qsort(sup, (size_t)K, sizeof(int64_t), by_index);
    } else {
      for (int64_t j = 0; j < K; ++j) sup[j] = j;
    }
    if (topk_idx && topk > 0)
      for (int64_t j = 0; j < K; ++j) topk_idx[t * K + j] = (int32_t)sup[j];

    /* log-softmax of both over the support */
    const double lse_a = logsumexp(a, sup, K);
    const double lse_b = logsumexp(b, sup, K);
    double fkl = 0.0, rkl = 0.0, ck = 0.0;
    for (int64_t j = 0; j < K; ++j) {
      const int64_t i = sup[j];
      const double lpt = a[i] - lse_a, lps = b[i] - lse_b;
      const double pt = exp(lpt), ps = exp(lps);
      fkl += pt * (lpt - lps);
      rkl += ps * (lps - lpt);
      ck += (pt + ps) * (1.0 + fabs(lpt) + fabs(lps));
    }
    /* conf: the full-vocabulary (softened) teacher probability of the label */
    const double conf = exp(a[labels[t]] - logsumexp(a, NULL, V));
    const double t2 = tau * tau;
    double loss;
    if (kd_type == KD_KL) loss = t2 * fkl;
    else if (kd_type == KD_RKL) loss = t2 * rkl;
    else if (kd_type == KD_CAKLD) loss = t2 * (conf * rkl + (1.0 - conf) * fkl);
    else {
      double se = 0.0;
      for (int64_t i = 0; i < V; ++i) {
        const double d = bf16v(srow[i]) - bf16v(trow[i]);
        se += d * d;
      }
      loss = se / (double)V;
      cond[2 * t + 1] = loss;
    }
    tk[0] = loss;
    tk[1] = t2 * fkl;
    tk[2] = t2 * rkl;
    cond[2 * t] = t2 * ck;

    if (dstudent || gmag) {
      if (kd_type == KD_MSE) {
        for (int64_t i = 0; i < V; ++i) {
          const double g = gs * 2.0 * (bf16v(srow[i]) - bf16v(trow[i])) / (double)V;
          if (dstudent) dstudent[t * V + i] = g;
          if (gmag) gmag[t * V + i] = fabs(g);
        }
      } else {
        /* d(tau^2 KL(a, b = s / tau)) / ds = tau * dKL / db */
        const double wf = kd_type == KD_KL ? 1.0 : kd_type == KD_RKL ? 0.0 : 1.0 - conf;
        const double wr = kd_type == KD_KL ? 0.0 : kd_type == KD_RKL ? 1.0 : conf;
        for (int64_t j = 0; j < K; ++j) {
          const int64_t i = sup[j];
          const double lpt = a[i] - lse_a, lps = b[i] - lse_b;
          const double pt = exp(lpt), ps = exp(lps);
          const double g = gs * tau * (wf * (ps - pt) + wr * ps * ((lps - lpt) - rkl));
          if (dstudent) dstudent[t * V + i] = g;
          if (gmag) gmag[t * V + i] = fabs(gs * tau) * (pt + ps) * (1.0 + fabs(lps - lpt) + fabs(rkl));
        }
      }
    }
    free(a);
    free(b);
    free(sup);
  }
  if (fail) return 2;

  losses[0] = losses[1] = losses[2] = 0.0;
  if (n_valid) {
    for (int64_t t = 0; t < T; ++t)
      for (int k = 0; k < 3; ++k) losses[k] += tok[3 * t + k];
    for (int k = 0; k < 3; ++k) losses[k] /= (double)n_valid;
  }
  return 0;
}
