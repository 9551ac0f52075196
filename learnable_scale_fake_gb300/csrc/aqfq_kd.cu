// aqfq_kd.cu -- distillation losses between student and teacher logits
// (forward KL, reverse KL, cakld, mse; whole vocabulary or the teacher's
// top-K support; temperature) with the gradient for the student logits.
//
// The operation (AngelSlim "QAT + DeepSpeed ZeRO-3" page, table "KD variants
// (loss_type)" and the cakld formula; mcore_qad article, section 2.5, top-k
// distillation without a [tokens, vocab] tensor): per position with a valid
// label, with a = teacher / tau and b = student / tau over the support U
// (every token, or the teacher's K largest logits):
//   p_t = softmax_U(a), p_s = softmax_U(b)
//   fkl = sum p_t (log p_t - log p_s),  rkl = sum p_s (log p_s - log p_t)
//   conf = softmax(a)[label] over the whole vocabulary
//   loss = tau^2 fkl | tau^2 rkl | tau^2 (conf rkl + (1 - conf) fkl) | mean (s - t)^2
// averaged over the valid positions; the gradient of that mean times
// grad_scale is written for the student logits.
//
// Layout of the work: one cluster of 8 CTAs per position (persistent over
// positions), 256 threads each: three CTAs per SM for the whole vocabulary of
// a Qwen3-sized model.  CTA r holds the vocabulary slice [r S, r S + S) of
// both rows in shared memory, brought in by two bulk copies (TMA, mbarrier)
// issued as soon as the previous position has released the buffer, so HBM
// sees each logit once and each gradient element once; the other CTAs of the
// SM compute while one waits.  The row statistics (max and sum of
// exponentials) and the top-K histograms are combined across the cluster
// through distributed shared memory in a fixed order, so every CTA holds
// bit-identical row values; each slice's loss sums go to the workspace and
// a second kernel adds them in rank order: results are reproducible.
// The top-K loss depends on the student only on the support, and its
// selection state fits one CTA: up to 2^19 vocabulary entries it runs one
// CTA per position (kd_topk_row_kernel, block barriers only); beyond that in
// the cluster kernel, whose CTAs then copy the teacher's slice alone and load
// the student's vectors that hold support elements from device memory.
//
// Top-K support: 16-bit order-preserving keys of the teacher's BF16 values.
// The K-th largest element is at least the K-th largest of the 8-element
// vector maxima, so a histogram of vector maxima (one count per vector)
// bounds the threshold from below; only elements above that bound are
// counted at 12-bit resolution, then the threshold bin is resolved to the
// exact key with a 4-bit histogram; equal keys are taken in index order.
//
// Numerics: logits are scaled to base-2 units (x = v * log2(e) / tau) and
// exponentials use ex2.approx; log-sum-exp uses the maximum.  The loss is
// summed per element as p_t d - p_t + p_s (forward) and -p_s d - p_s + p_t
// (reverse), d = log p_t - log p_s in nats: the added -p_t + p_s terms sum to
// zero exactly in real arithmetic and make the sum insensitive, to first
// order, to the rounding of the two normalisers.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "aqfq.h"
#include "aqfq_internal.h"
#include "aqfq_sm100.cuh"

namespace aqfq {
namespace {

using sm100::smem_u32;

#ifndef AQFQ_KD_CLUSTER
#define AQFQ_KD_CLUSTER 8
#endif
#ifndef AQFQ_KD_NBUF
#define AQFQ_KD_NBUF 1
#endif
constexpr int kCl = AQFQ_KD_CLUSTER;  // CTAs per position (vocabulary slices)
constexpr int kNbuf = AQFQ_KD_NBUF;   // slice buffers per CTA
static_assert(kNbuf == 1, "positions handed out one at a time use one slice buffer");
#ifndef AQFQ_KD_THREADS
#define AQFQ_KD_THREADS 256
#endif
constexpr int kThr = AQFQ_KD_THREADS;  // threads per CTA
#ifndef AQFQ_KD_MINB
#define AQFQ_KD_MINB (AQFQ_KD_THREADS <= 256 ? 3 : 2)
#endif
constexpr int kMinBlocks = AQFQ_KD_MINB;  // CTAs per SM the register budget is sized for
constexpr int kWarps = kThr / 32;
constexpr int kHist1 = 4096;    // bins: the top 12 bits of the 16-bit teacher key
constexpr int kHistWords = kHist1 / 2;  // two 16-bit counters per word (a slice has < 2^16 elements)
constexpr int kMaxPer = 256;  // top-K row kernel: vectors per thread, at most (V <= 2^19)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

struct KdArgs {
  const uint16_t* s;        // student [T, V] BF16
  const uint16_t* t;        // teacher [T, V] BF16
  const int32_t* labels;    // [T]
  int32_t* ws_head;         // [0]: number of valid positions, [1]: error word
  const int64_t* rows;      // [T]: the valid positions ascending, then the ignored ones
  unsigned long long* ticket;  // the next position ticket (zeroed by the count kernel)
  float* part;              // workspace [T, kCl, 2]: each slice's forward / reverse KL sums
  float* rowx;              // workspace [T, 2]: conf and the sum of (s - t)^2 of each position
  uint16_t* ds;             // optional [T, V] BF16
  int32_t* topk_idx;        // optional [T, K]
  int64_t T, V;
  int32_t S;                // slice length, a multiple of 8
  int32_t K;                // 0: whole vocabulary
  int32_t type;             // AQFQ_KD_*
  float ks;                 // log2(e) / tau
  float tau, tau2, grad_scale;
};

// Per-CTA bookkeeping, kept small: with the Qwen3-sized vocabulary the
// whole-vocabulary layout (slices + this) fits three CTAs per SM when the
// thread count allows it.
struct __align__(16) KdShared {
  uint64_t full[2];         // mbarriers of the two slice buffers
  unsigned long long tk0;   // rank 0: the cluster's first position ticket
  unsigned long long tk;    // the ticket received in the last exchange that carried one
  float xw[2][12];          // this CTA's reduction record (alternating exchange slots, 48 B
                            // each; words 10-11: rank 0's next position ticket)
  float red[kWarps][9];     // per-warp records; per-warp loss sums in [w][0..1]
  int32_t ired[kWarps + 1];
  int32_t sel[8];           // threshold search results
  int32_t err;
  float res[10];            // the last reduction's result, for every thread
};

static_assert(offsetof(KdShared, xw) % 16 == 0 && sizeof(KdShared::xw[0]) % 16 == 0,
              "exchange slots are read with 16-byte remote loads");

// top-K only (dynamic shared memory after the histograms)
struct __align__(16) TopkShared {
  uint32_t hist2[16];       // low nibble of the keys in the threshold bin
  uint32_t h2all[kCl][16];  // hist2 of every rank
  uint32_t bins[8 * (kThr / kCl)];  // cluster-wide counts of one search step's bins
};

// ---------------------------------------------------------------------------
// cluster primitives (PTX: barrier.cluster, mapa, ld.shared::cluster)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; orders shared-memory writes before
// the barrier with reads by any CTA after it
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t remote_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_remote_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
// 16 bytes (four words) from a 16-byte aligned shared::cluster address
__device__ __forceinline__ uint4 ld_remote_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
// 8 bytes (two words) from an 8-byte aligned shared::cluster address
__device__ __forceinline__ uint2 ld_remote_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_remote_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// one bulk copy global -> this CTA's shared memory, completing on `bar`
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// arithmetic helpers (f2 pairs and their packed f32x2 operations come from
// the device header)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ f2 ex2x2(f2 v) { return mk2(ex2(lo2(v)), ex2(hi2(v))); }
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// largest of the 8 BF16 values of a vector, as binary32
__device__ __forceinline__ float vmax8(uint4 w) {
  const uint32_t m = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}
// order-preserving 16-bit key of a BF16 value; -0 and +0 share a key
__device__ __forceinline__ uint32_t okey(uint32_t b) {
  b &= 0xFFFFu;
  if (b == 0x8000u) b = 0;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ uint32_t word(const uint4& w, int i) {
  return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}
__device__ __forceinline__ uint32_t key_of(const uint4& w, int j) {
  const uint32_t x = word(w, j >> 1);
  return okey(j & 1 ? x >> 16 : x);
}
// key of a binary32 value that is exactly a BF16 value
__device__ __forceinline__ uint32_t key_of_f(float f) { return okey(__float_as_uint(f) >> 16); }
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// A set of logits v, kept in raw (BF16) units so that every exponent is a
// difference of nearby values: m = max v, z = sum 2^((v - m) ks), b = a
// weighted sum under the same weights; z == 0 marks an empty set.
struct Online {
  float m, z, b;
};
__device__ __forceinline__ Online online_empty() { return Online{-INFINITY, 0.0f, 0.0f}; }
// symmetric in its operands (bit for bit), so butterfly lanes agree
__device__ __forceinline__ Online online_merge(Online a, Online c, float ks) {
  const float m = fmaxf(a.m, c.m);
  const float fa = a.z != 0.0f ? ex2(__fmul_rn(__fsub_rn(a.m, m), ks)) : 0.0f;
  const float fc = c.z != 0.0f ? ex2(__fmul_rn(__fsub_rn(c.m, m), ks)) : 0.0f;
  return Online{m, __fadd_rn(__fmul_rn(a.z, fa), __fmul_rn(c.z, fc)),
                __fadd_rn(__fmul_rn(a.b, fa), __fmul_rn(c.b, fc))};
}
__device__ __forceinline__ Online online_shfl(Online a, int d) {
  return Online{__shfl_xor_sync(0xFFFFFFFFu, a.m, d), __shfl_xor_sync(0xFFFFFFFFu, a.z, d),
                __shfl_xor_sync(0xFFFFFFFFu, a.b, d)};
}

// Waits until the phase of `bar` with the given parity completes.  The thread
// sleeps in mbarrier.try_wait (no polling loop issuing instructions); gives
// up after about 2^31 clock cycles (~1 s) and returns false.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > (1ll << 31)) return false;
  }
}

// A reduction record: online states of teacher and student, two sums and one
// integer combined by max (KMAX) or by sum.
struct Rec {
  Online t, s;
  float u, v;
  int k;
};
__device__ __forceinline__ Rec rec_empty() { return Rec{online_empty(), online_empty(), 0.0f, 0.0f, 0}; }
template <bool KMAX>
__device__ __forceinline__ Rec rec_merge(const Rec& a, const Rec& c, float ks) {
  return Rec{online_merge(a.t, c.t, ks), online_merge(a.s, c.s, ks), __fadd_rn(a.u, c.u),
             __fadd_rn(a.v, c.v), KMAX ? max(a.k, c.k) : a.k + c.k};
}
__device__ __forceinline__ Rec rec_shfl(const Rec& a, int d) {
  return Rec{online_shfl(a.t, d), online_shfl(a.s, d), __shfl_xor_sync(0xFFFFFFFFu, a.u, d),
             __shfl_xor_sync(0xFFFFFFFFu, a.v, d), __shfl_xor_sync(0xFFFFFFFFu, a.k, d)};
}
// xor butterfly over the first N lanes (N a power of two, at most 32): each
// of them ends with the same total (the merge is symmetric bit for bit), in a
// fixed order.  Merging an empty record is exact (a scale of 2^0 = 1 and a
// zero term), so with lanes N.. empty this gives the bits of the full
// 32-lane butterfly in log2(N) steps.
template <bool KMAX, int N = 32>
__device__ __forceinline__ Rec warp_rec(Rec a, float ks) {
  static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "a power of two up to 32");
#pragma unroll
  for (int d = N / 2; d >= 1; d >>= 1) a = rec_merge<KMAX>(a, rec_shfl(a, d), ks);
  return a;
}
__device__ __forceinline__ void rec_store(float* p, const Rec& a) {
  p[0] = a.t.m; p[1] = a.t.z; p[2] = a.t.b; p[3] = a.s.m; p[4] = a.s.z; p[5] = a.s.b;
  p[6] = a.u; p[7] = a.v; p[8] = __int_as_float(a.k);
}
__device__ __forceinline__ Rec rec_load(const float* p) {
  return Rec{Online{p[0], p[1], p[2]}, Online{p[3], p[4], p[5]}, p[6], p[7], __float_as_int(p[8])};
}

// Cluster reduction of one record per warp (`wr`: the warp's total, the same in
// every lane).  Warp 0 merges the warps' records into the CTA's record and
// puts it in this CTA's exchange slot `par`; the cluster synchronises; warp 0
// of every CTA reads the kCl CTA records (lane r from rank r), merges them in
// a fixed order and broadcasts the total through shared memory, so all CTAs
// hold bit-identical totals.  k_before (if not NULL) receives the sum of k
// over the ranks below this one.  With `tick` (not NULL) the exchange also
// carries rank 0's *tick (next position ticket) to every CTA's *tick.  A slot is rewritten two exchanges later,
// after a barrier that every CTA passes only once it has read the slot; the
// warp records and the result are rewritten only after barriers that every
// thread reaches after reading them.
template <bool KMAX>
__device__ __forceinline__ Rec cluster_rec(const Rec& wr, KdShared* sh, int& par, float ks,
                                           int* k_before = nullptr,
                                           unsigned long long* tick = nullptr) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) rec_store(sh->red[w], wr);
  __syncthreads();
  if (w == 0) {
    Rec x = l < kWarps ? rec_load(sh->red[l]) : rec_empty();
    x = warp_rec<KMAX, kWarps>(x, ks);
    if (l == 0) {
      rec_store(sh->xw[par], x);
      if (tick) {
        sh->xw[par][10] = __uint_as_float(uint32_t(*tick));
        sh->xw[par][11] = __uint_as_float(uint32_t(*tick >> 32));
      }
    }
  }
  cluster_sync();
  if (w == 0) {
    Rec x = rec_empty();
    if (l < kCl) {  // the record in two 16-byte loads and one word
      const uint32_t base = remote_addr(&sh->xw[par][0], uint32_t(l));
      const uint4 a0 = ld_remote_v4(base), a1 = ld_remote_v4(base + 16u);
      const float v[9] = {__uint_as_float(a0.x), __uint_as_float(a0.y), __uint_as_float(a0.z),
                          __uint_as_float(a0.w), __uint_as_float(a1.x), __uint_as_float(a1.y),
                          __uint_as_float(a1.z), __uint_as_float(a1.w), ld_remote_f32(base + 32u)};
      x = rec_load(v);
      if (tick && l == 0) {  // rank 0's ticket
        const uint2 t = ld_remote_v2(base + 40u);
        sh->tk = (static_cast<unsigned long long>(t.y) << 32) | t.x;
      }
    }
    if (k_before) {  // exclusive prefix over the ranks below this one
      int inc = x.k;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (l >= d) inc += y;
      }
      if (uint32_t(l) == cluster_rank()) sh->res[9] = __int_as_float(inc - x.k);
    }
    x = warp_rec<KMAX, kCl>(x, ks);
    if (l == 0) rec_store(sh->res, x);
  }
  __syncthreads();
  const Rec r = rec_load(sh->res);
  if (k_before) *k_before = __float_as_int(sh->res[9]);
  if (tick) *tick = sh->tk;
  par ^= 1;
  return r;
}

// Block-wide inclusive scan of one int per thread; returns (inclusive, total).
__device__ __forceinline__ int block_scan(int v, int& total, KdShared* sh) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
    if (l >= d) x += y;
  }
  if (l == 31) sh->ired[w] = x;
  __syncthreads();
  int before = 0;
  total = 0;
  for (int k = 0; k < kWarps; ++k) {
    if (k < w) before += sh->ired[k];
    total += sh->ired[k];
  }
  __syncthreads();
  return x + before;
}

// After a cluster barrier: walking down from bin `top`, the bin at which the
// cluster-wide count of a 4096-bin histogram (16-bit counters, bin b in half
// b & 1 of word b >> 1) reaches K, and the count above
// that bin.  Returns false (bin 0, the whole count) when the histogram holds
// fewer than K.  All threads call it.  A step covers 8 * kThr / kCl bins (256
// with 256 threads and 8 ranks) in aligned blocks of 8: thread t loads block
// t / kCl of the step from rank t % kCl (one 16-byte remote load), the kCl
// threads of a block add their counts, and one warp scans the step's bins
// from the top.  Steps start at the top of `top`'s block (bins above `top`
// are empty).
__device__ __forceinline__ bool find_from_top(const uint32_t* hist, int top, int K, int& bin,
                                              int& above, KdShared* sh, TopkShared* tk) {
  constexpr int kBlocks = kThr / kCl;  // 8-bin blocks per step
  constexpr int kStep = 8 * kBlocks;
  static_assert(kThr % kCl == 0 && 32 % kCl == 0, "the ranks of a block share a warp");
  static_assert(kStep % 32 == 0 && kStep <= 1024, "the scanning warp takes kStep / 32 bins per lane");
  constexpr int kPer = kStep / 32;  // bins per lane of the scanning warp
  const int tid = threadIdx.x, j = tid / kCl, r = tid % kCl;
  int base = 0;
  for (int hi = top | 7; hi >= 0; hi -= kStep) {
    const int bh = hi - 8 * j;  // this block: bins [bh - 7, bh]; bh % 8 == 7
    uint32_t c[8];              // c[i]: bin bh - i
    {
      uint4 w = make_uint4(0, 0, 0, 0);
      if (bh >= 0) w = ld_remote_v4(remote_addr(hist + ((bh - 7) >> 1), uint32_t(r)));
      const uint32_t q[4] = {w.x, w.y, w.z, w.w};  // word m holds bins bh-7+2m (low), bh-6+2m (high)
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = (q[(7 - i) >> 1] >> (((7 - i) & 1) * 16)) & 0xFFFFu;
    }
#pragma unroll
    for (int d = kCl / 2; d >= 1; d >>= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] += __shfl_xor_sync(0xFFFFFFFFu, c[i], d);
    if (r == 0)
#pragma unroll
      for (int i = 0; i < 8; ++i) tk->bins[8 * j + i] = c[i];  // step index 8 j + i = bin hi - (8 j + i)
    __syncthreads();
    if (tid < 32) {  // lane l: step indices [kPer l, kPer l + kPer), from the top down
      uint32_t v[kPer];
      int cl = 0;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        v[i] = tk->bins[kPer * tid + i];
        cl += int(v[i]);
      }
      int x = cl;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
        if (tid >= d) x += y;
      }
      const int incl = base + x;
      if (incl - cl < K && incl >= K) {  // the crossing lies in this lane's bins
        int run = incl - cl;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          if (run + int(v[i]) >= K) {
            sh->sel[6] = hi - (kPer * tid + i);
            sh->sel[7] = run;
            break;
          }
          run += int(v[i]);
        }
      }
      if (tid == 31) sh->sel[1] = incl;  // running total after this step
    }
    __syncthreads();
    base = sh->sel[1];
    if (base >= K) {
      bin = sh->sel[6];
      above = sh->sel[7];
      __syncthreads();
      return true;
    }
    __syncthreads();
  }
  bin = 0;
  above = base;
  return false;
}

// Block reduction of one record per warp (`wr`: the warp's total, the same in
// every lane): warp 0 merges the warps' records in warp order; every thread
// receives the total.
template <bool KMAX>
__device__ __forceinline__ Rec block_rec(const Rec& wr, KdShared* sh, float ks) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) rec_store(sh->red[w], wr);
  __syncthreads();
  if (w == 0) {
    Rec x = l < kWarps ? rec_load(sh->red[l]) : rec_empty();
    x = warp_rec<KMAX, kWarps>(x, ks);
    if (l == 0) rec_store(sh->res, x);
  }
  __syncthreads();
  const Rec r = rec_load(sh->res);
  __syncthreads();  // the records are rewritten by the next reduction
  return r;
}

// Walking down from bin `top` of this CTA's 4096-bin histogram of 32-bit
// counters: the bin at which the count reaches K and the count above it.
// Warp 0 scans 256 bins per step (8 per lane); every thread receives the
// result.  Returns false (bin 0, the whole count) when the histogram holds
// fewer than K.  All threads call it.
__device__ __forceinline__ bool find_local(const uint32_t* hist, int top, int K, int& bin,
                                           int& above, KdShared* sh) {
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    int base = 0, found = 0, fb = 0, fa = 0;
    for (int hi = top; hi >= 0 && !found; hi -= 256) {
      uint32_t c[8];  // c[i]: bin hi - 8 l - i
      int cl = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int b = hi - 8 * l - i;
        c[i] = b >= 0 ? hist[b] : 0u;
        cl += int(c[i]);
      }
      int x = cl;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
        if (l >= d) x += y;
      }
      const int incl = base + x;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, incl - cl < K && incl >= K);
      if (m) {
        const int src = __ffs(m) - 1;
        if (l == src) {
          int run = incl - cl;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (run + int(c[i]) >= K) {
              fb = hi - 8 * l - i;
              fa = run;
              break;
            }
            run += int(c[i]);
          }
        }
        fb = __shfl_sync(0xFFFFFFFFu, fb, src);
        fa = __shfl_sync(0xFFFFFFFFu, fa, src);
        found = 1;
      }
      base = __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (l == 0) {
      sh->sel[1] = found;
      sh->sel[6] = found ? fb : 0;
      sh->sel[7] = found ? fa : base;
    }
  }
  __syncthreads();
  bin = sh->sel[6];
  above = sh->sel[7];
  const bool ok = sh->sel[1] != 0;
  __syncthreads();  // sel is rewritten next
  return ok;
}

// 16 bytes of a logit row from device memory (read-only for the kernel)
__device__ __forceinline__ uint4 ld_row16(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Visits the vectors listed in cand[0..nc) (ascending vector indices) and calls
// emit(local index, position) for every element that satisfies pred(local
// index, key); the position counts those elements from 0 in index order.
// All threads call it.
template <class Pred, class Emit>
__device__ __forceinline__ void ordered_scan(const uint16_t* tsl, const uint16_t* cand, int nc,
                                             Pred pred, Emit emit, KdShared* sh) {
  int base = 0;
  for (int p0 = 0; p0 < nc; p0 += kThr) {
    const int p = p0 + int(threadIdx.x);
    uint32_t m8 = 0;
    int v = 0;
    if (p < nc) {
      v = cand[p];
      const uint4 w = *reinterpret_cast<const uint4*>(tsl + 8 * v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (pred(8 * v + j, key_of(w, j))) m8 |= 1u << j;
    }
    const int c = __popc(m8);
    int total;
    int pos = base + block_scan(c, total, sh) - c;
    while (m8) {
      const int j = __ffs(m8) - 1;
      emit(8 * v + j, pos++);
      m8 &= m8 - 1;
    }
    base += total;
  }
}

// One cluster per position, persistent over positions.
//   TOPK   restrict to the teacher's top-K support
//   RGRAD  the gradient has a reverse-KL part (rkl, cakld): pass 1 also sums
//          2^(x_s - m) (x_s - x_t) for the reverse KL that centres it
//   MSE    mean squared error loss and gradient
template <bool TOPK, bool RGRAD, bool MSE>
__global__ void __launch_bounds__(kThr, kMinBlocks) kd_loss_kernel(const KdArgs a) {
  extern __shared__ __align__(16) uint8_t kd_smem[];
  KdShared* sh = reinterpret_cast<KdShared*>(kd_smem);
  const int nvb = TOPK ? (a.S / 8 + 7) / 8 * 8 : 0;  // vector slots, padded to 16 bytes
  uint32_t* vhist = reinterpret_cast<uint32_t*>(kd_smem + sizeof(KdShared));  // vector-max bins
  uint32_t* hist1 = vhist + (TOPK ? kHistWords : 0);                           // element bins
  TopkShared* tk = reinterpret_cast<TopkShared*>(hist1 + (TOPK ? kHistWords : 0));
  uint16_t* vbin = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(tk) +
                                               (TOPK ? sizeof(TopkShared) : 0));  // bin of each vector max
  uint16_t* cand = vbin + nvb;                                                 // candidate vectors
  // kNbuf buffers of [teacher S | student S]; the top-K loss reads the
  // student only on the support, from device memory, so its buffers hold the
  // teacher's slice alone
  uint16_t* buf0 = cand + nvb;
  constexpr int kRows = TOPK ? 1 : 2;  // logit rows per buffer
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int64_t v0 = int64_t(rank) * a.S;  // first vocabulary index of this slice
  int64_t n64 = a.V - v0;
  if (n64 > a.S) n64 = a.S;
  if (n64 < 0) n64 = 0;
  const int nvec = int(n64) >> 3;  // V % 8 == 0 and S % 8 == 0
  const uint32_t bytes = uint32_t(n64) * 2u;
  const int nval = a.ws_head[0];
  const float ks = a.ks;
  // d(tau^2 KL(s / tau)) / ds = tau dKL/db, over the mean
  const float gsc = nval > 0 ? (MSE ? a.grad_scale * 2.0f / (float(a.V) * float(nval))
                                    : a.grad_scale * a.tau / float(nval))
                             : 0.0f;
  if (tid == 0) {
    sm100::mbar_init(&sh->full[0], 1);
    sm100::mbar_init(&sh->full[1], 1);
    sh->err = 0;
    sm100::fence_barrier_init();
  }
  if (TOPK) {
    for (int i = tid; i < 2 * kHistWords; i += kThr) vhist[i] = 0;
    if (tid < 16) tk->hist2[tid] = 0;
  }
  __syncthreads();

  auto prefetch = [&](int64_t r, int b) {  // thread 0
    uint16_t* tb = buf0 + size_t(b) * kRows * a.S;
    if (bytes) {
      sm100::mbar_arrive_expect_tx(&sh->full[b], uint32_t(kRows) * bytes);
      bulk_load(tb, a.t + r * a.V + v0, bytes, &sh->full[b]);
      if (!TOPK) bulk_load(tb + a.S, a.s + r * a.V + v0, bytes, &sh->full[b]);
    } else {
      sm100::mbar_arrive(&sh->full[b]);  // an empty slice completes the phase at once
    }
  };
  // Valid positions are handed out at run time, so that clusters on busier
  // SMs take fewer: ticket t is the t-th valid position of the list.  Rank 0
  // takes the cluster's next ticket while a position runs and passes it to
  // its peers in that position's first exchange; the first one through a
  // cluster barrier.  Every CTA of a cluster holds the same tickets.
  if (tid == 0 && rank == 0) sh->tk0 = atomicAdd(a.ticket, 1ull);
  cluster_sync();
  unsigned long long tcur;
  {
    const uint2 t = ld_remote_v2(remote_addr(&sh->tk0, 0u));
    tcur = (static_cast<unsigned long long>(t.y) << 32) | t.x;
  }
  if (tid == 0 && tcur < (unsigned long long)nval) prefetch(a.rows[tcur], 0);
  uint32_t uses[2] = {0, 0};
  int it = 0, par = 0;

  while (tcur < (unsigned long long)nval) {
    const int64_t row = a.rows[tcur];
    unsigned long long tnext = 0;  // the next ticket: rank 0 takes it now
    if (tid == 0 && rank == 0) tnext = atomicAdd(a.ticket, 1ull);
    uint16_t* drow = a.ds ? a.ds + row * a.V + v0 : nullptr;
    const int b = 0;
    ++it;
    if (!wait_phase(&sh->full[b], uses[b] & 1u)) atomicExch(&sh->err, 1);
    ++uses[b];
    const uint16_t* tsl = buf0 + size_t(b) * kRows * a.S;
    const uint4* t4 = reinterpret_cast<const uint4*>(tsl);
    // the student's 8-element vector v of this slice: shared memory, or (top-K
    // support) device memory; rows and slices start on 16-byte boundaries
    const uint4* s4 = reinterpret_cast<const uint4*>(tsl + a.S);
    const uint4* s4g = reinterpret_cast<const uint4*>(a.s + row * a.V + v0);
    auto svec = [&](int v) -> uint4 { return TOPK ? __ldg(s4g + v) : s4[v]; };
    const int64_t lloc = int64_t(a.labels[row]) - v0;  // the label's index within the slice

    // ---- pass 1: whole-vocabulary statistics (teacher; student unless TOPK) --
    // One read of each vector: per-thread running maxima (raw units), the
    // sums of 2^((v - max) ks) rescaled when a vector raises them; warps then
    // merge by butterfly and the cluster merges the warps' records.
    float tmax = -INFINITY, smax = -INFINITY;  // raw (BF16) maxima: the sums' reference
    f2 zt = 0, zs = 0, bb = 0, se2 = 0;
    {
      const f2 KS = mk2(ks, ks);
      for (int v = tid; v < nvec; v += kThr) {
        const uint4 w = t4[v];
        const float vt = vmax8(w);
        if (TOPK) {
          const uint32_t kb = key_of_f(vt) >> 4;
          vbin[v] = uint16_t(kb);
          atomicAdd(&vhist[kb >> 1], 1u << ((kb & 1u) * 16));
        }
        if (vt > tmax) {
          const float f = ex2(__fmul_rn(__fsub_rn(tmax, vt), ks));
          zt = mul2(zt, mk2(f, f));
          tmax = vt;
        }
        const f2 TM = mk2(tmax, tmax);
        uint4 x = make_uint4(0, 0, 0, 0);
        f2 SM = 0;
        if (!TOPK) {
          x = svec(v);
          const float vs = vmax8(x);
          if (vs > smax) {
            const float f = ex2(__fmul_rn(__fsub_rn(smax, vs), ks));
            zs = mul2(zs, mk2(f, f));
            if (RGRAD) bb = mul2(bb, mk2(f, f));
            smax = vs;
          }
          SM = mk2(smax, smax);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const f2 t2 = bf2(word(w, i));
          zt = add2(zt, ex2x2(mul2(sub2(t2, TM), KS)));
          if (!TOPK) {
            const f2 s2 = bf2(word(x, i));
            const f2 es = ex2x2(mul2(sub2(s2, SM), KS));
            zs = add2(zs, es);
            if (RGRAD || MSE) {
              const f2 d = sub2(s2, t2);
              if (RGRAD) bb = fma2(es, d, bb);
              if (MSE) se2 = fma2(d, d, se2);
            }
          }
        }
      }
    }
    // the label's teacher logit (raw), from the thread whose vectors hold it
    const bool owns_label = lloc >= 0 && lloc < n64 && int((lloc >> 3) % kThr) == tid;
    const float xl = owns_label ? __uint_as_float(uint32_t(tsl[lloc]) << 16) : 0.0f;
    const Rec mine{Online{tmax, __fadd_rn(lo2(zt), hi2(zt)), 0.0f},
                   Online{smax, __fadd_rn(lo2(zs), hi2(zs)), __fmul_rn(__fadd_rn(lo2(bb), hi2(bb)), ks)},
                   __fadd_rn(lo2(se2), hi2(se2)), 0.0f,
                   (TOPK && tmax > -INFINITY) ? int(key_of_f(tmax)) : 0};
    Rec wr = warp_rec<true>(mine, ks);
    {  // the label's value: one thread of one CTA holds it; the butterfly adds zeros
      float x = xl;
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, d));
      wr.v = x;
    }
    const Rec R1 = cluster_rec<true>(wr, sh, par, ks, nullptr, &tnext);
    const Online T_ = R1.t, S_ = R1.s;
    const float SE = R1.u, XL = R1.v;
    const int kmax = R1.k;
    // conf: the whole-vocabulary teacher probability of the label
    const float conf = ex2(__fmaf_rn(__fsub_rn(XL, T_.m), ks, -log2f(T_.z)));

    // ---- top-K support: threshold key, ties by index ----------------------
    uint32_t tkey = 0;
    int idx_lim = -1, tbin = 0, nc = 0;
    if (TOPK) {
      const int top = kmax >> 4;
      int b0 = 0, above = 0;
      if (!find_from_top(vhist, top, a.K, b0, above, sh, tk)) b0 = 0;
      // keys at or above the bound span few 12-bit bins: count exact 16-bit
      // keys there (one histogram gives the threshold key and the per-rank
      // ties); otherwise 12-bit bins, then the low 4 bits of the threshold bin
      const bool exact = (top - b0 + 1) * 16 <= kHist1;
      const uint32_t kbase = uint32_t(b0) << 4;
      {  // candidate vectors (maximum at or above the bound), ascending: a
         // contiguous range of vectors per thread and one block scan
        const int per = (nvec + kThr - 1) / kThr, v0t = tid * per;
        const int v1t = min(nvec, v0t + per);
        int c = 0;
        for (int v = v0t; v < v1t; ++v) c += int(vbin[v]) >= b0;
        int total;
        int pos = block_scan(c, total, sh) - c;
        for (int v = v0t; v < v1t; ++v)
          if (int(vbin[v]) >= b0) cand[pos++] = uint16_t(v);
        nc = total;
        __syncthreads();
      }
      // elements at or above the bound: exact-key or 12-bit histogram
      for (int p = tid; p < nc; p += kThr) {
        const uint4 w = t4[cand[p]];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t k = key_of(w, j);
          if (int(k >> 4) >= b0) {
            const uint32_t bin = exact ? k - kbase : (k >> 4);
            atomicAdd(&hist1[bin >> 1], 1u << ((bin & 1u) * 16));
          }
        }
      }
      __syncthreads();
      cluster_sync();
      if (exact) {
        int tb = 0;
        find_from_top(hist1, int((uint32_t(top + 1) << 4) - 1 - kbase), a.K, tb, above, sh, tk);
        const int need = a.K - above;  // elements equal to the threshold key to take
        if (tid < kCl)
          tk->h2all[tid][0] =
              (ld_remote_u32(remote_addr(hist1 + (tb >> 1), uint32_t(tid))) >> ((tb & 1) * 16)) & 0xFFFFu;
        __syncthreads();
        if (tid == 0) {
          int before = 0;
          for (uint32_t r = 0; r < rank; ++r) before += int(tk->h2all[r][0]);
          const int eq = int(tk->h2all[rank][0]);
          int take = need - before;
          take = take < 0 ? 0 : (take > eq ? eq : take);
          sh->sel[2] = int(kbase + uint32_t(tb));
          sh->sel[3] = take;
          sh->sel[4] = eq;
          sh->sel[5] = -1;
        }
        __syncthreads();
      } else {
      int bstar = 0;
      find_from_top(hist1, top, a.K, bstar, above, sh, tk);  // holds at least K
      const int need = a.K - above;
      for (int p = tid; p < nc; p += kThr) {
        const int v = cand[p];
        if (int(vbin[v]) < bstar) continue;
        const uint4 w = t4[v];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t k = key_of(w, j);
          if (int(k >> 4) == bstar) atomicAdd(&tk->hist2[k & 15u], 1u);
        }
      }
      __syncthreads();
      cluster_sync();
      if (tid < kCl * 16)
        tk->h2all[tid >> 4][tid & 15] = ld_remote_u32(remote_addr(&tk->hist2[tid & 15], tid >> 4));
      __syncthreads();
      if (tid == 0) {
        int cum = 0, l = 15;
        for (; l > 0; --l) {
          int h = 0;
          for (int r = 0; r < kCl; ++r) h += int(tk->h2all[r][l]);
          if (cum + h >= need) break;
          cum += h;
        }
        const int q = need - cum;  // elements equal to the threshold key to take
        int before = 0;
        for (uint32_t r = 0; r < rank; ++r) before += int(tk->h2all[r][l]);
        const int eq = int(tk->h2all[rank][l]);
        int take = q - before;
        take = take < 0 ? 0 : (take > eq ? eq : take);
        sh->sel[2] = int((uint32_t(bstar) << 4) | uint32_t(l));
        sh->sel[3] = take;
        sh->sel[4] = eq;
        sh->sel[5] = -1;
      }
      __syncthreads();
      }
      tkey = uint32_t(sh->sel[2]);
      tbin = int(tkey >> 4);
      const int take = sh->sel[3], eq = sh->sel[4];
      if (take == eq) {
        idx_lim = 8 * nvec;
      } else if (take > 0) {  // the take-th equal element in index order
        ordered_scan(
            tsl, cand, nc, [&](int, uint32_t k) { return k == tkey; },
            [&](int i, int pos) {
              if (pos + 1 == take) sh->sel[5] = i;
            },
            sh);
        __syncthreads();
        idx_lim = sh->sel[5];
      }
    }
    auto selected = [&](int i, uint32_t k) { return k > tkey || (k == tkey && i <= idx_lim); };

    // ---- statistics over the support -----------------------------------------
    // each distribution over the support as (raw maximum M, L = log2 of the
    // sum of 2^((v - M) ks)): log2 p = (v - M) ks - L
    float m_t, m_s, l_t, l_s, bz;
    int sel_before = 0;
    if (TOPK) {
      Online ut = online_empty(), us = online_empty();
      int cnt = 0;
      for (int p = tid; p < nc; p += kThr) {
        const int v = cand[p];
        if (int(vbin[v]) < tbin) continue;
        const uint4 w = t4[v], x = svec(v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (!selected(8 * v + j, key_of(w, j))) continue;
          const uint32_t tw = word(w, j >> 1), sw = word(x, j >> 1);
          const float t = __uint_as_float(j & 1 ? tw & 0xFFFF0000u : tw << 16);
          const float s = __uint_as_float(j & 1 ? sw & 0xFFFF0000u : sw << 16);
          ut = online_merge(ut, Online{t, 1.0f, 0.0f}, ks);
          us = online_merge(us, Online{s, 1.0f, __fmul_rn(__fsub_rn(s, t), ks)}, ks);
          ++cnt;
        }
      }
      const Rec RS = cluster_rec<false>(warp_rec<false>(Rec{ut, us, 0.0f, 0.0f, cnt}, ks), sh, par,
                                        ks, &sel_before);
      m_t = RS.t.m;
      m_s = RS.s.m;
      l_t = log2f(RS.t.z);
      l_s = log2f(RS.s.z);
      bz = RS.s.b / RS.s.z;
    } else {
      m_t = T_.m;
      m_s = S_.m;
      l_t = log2f(T_.z);
      l_s = log2f(S_.z);
      bz = S_.b / S_.z;
    }

    // ---- pass 2: loss terms and the gradient ---------------------------------
    // dl = log2 of the normalisers' ratio (teacher over student), in base-2 units;
    // rkl0 = sum p_s (log p_s - log p_t) in nats (centres the reverse-KL gradient)
    const float dl = __fmaf_rn(__fsub_rn(m_t, m_s), ks, __fsub_rn(l_t, l_s));
    const float rkl0 = kLn2 * (bz + dl);
    const float wf = a.type == AQFQ_KD_KL ? 1.0f : a.type == AQFQ_KD_RKL ? 0.0f : 1.0f - conf;
    const float wr2 = a.type == AQFQ_KD_KL ? 0.0f : a.type == AQFQ_KD_RKL ? 1.0f : conf;
    const f2 KS = mk2(ks, ks), NLT = mk2(-l_t, -l_t), NLS = mk2(-l_s, -l_s);
    const f2 MT = mk2(m_t, m_t), MS = mk2(m_s, m_s);
    const float kl = ks * kLn2, ndl = -dl * kLn2;
    const f2 KL2 = mk2(kl, kl), NDL = mk2(ndl, ndl);
    // gradient: gsc (wf (p_s - p_t) - wr p_s (d + rkl)) = p_s (c - gsc wr d) - gsc wf p_t
    const f2 WF = mk2(gsc * wf, gsc * wf), NWF = mk2(-gsc * wf, -gsc * wf);
    const f2 NWR = mk2(-gsc * wr2, -gsc * wr2);
    const float c = gsc * wf - gsc * wr2 * rkl0;
    const f2 C2 = mk2(c, c), NGM = mk2(-gsc, -gsc);
    // the reverse sum: (p_t d - p_t + p_s) + (-p_s d - p_s + p_t) = -(p_s - p_t) d,
    // so it is formed from q = sum (p_s - p_t) d and the forward sum
    f2 fs2 = 0, q2 = 0;
    auto pass2_vector = [&](int v, bool masked) {
      const uint4 w = t4[v], x = svec(v);
      uint32_t out[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f2 t2 = bf2(word(w, i)), s2 = bf2(word(x, i));
        f2 pt = ex2x2(fma2(sub2(t2, MT), KS, NLT)), ps = ex2x2(fma2(sub2(s2, MS), KS, NLS));
        if (masked) {  // zero outside the support
          const bool in0 = selected(8 * v + 2 * i, key_of(w, 2 * i));
          const bool in1 = selected(8 * v + 2 * i + 1, key_of(w, 2 * i + 1));
          pt = mk2(in0 ? lo2(pt) : 0.0f, in1 ? hi2(pt) : 0.0f);
          ps = mk2(in0 ? lo2(ps) : 0.0f, in1 ? hi2(ps) : 0.0f);
        }
        const f2 d2 = sub2(t2, s2);
        const f2 dn = fma2(d2, KL2, NDL);  // log p_t - log p_s in nats
        const f2 diff = sub2(ps, pt);
        fs2 = add2(fs2, fma2(pt, dn, diff));
        q2 = fma2(diff, dn, q2);
        if (drow) {
          f2 g;
          if (MSE) g = mul2(d2, NGM);
          else if (RGRAD) g = fma2(ps, fma2(NWR, dn, C2), mul2(NWF, pt));
          else g = mul2(WF, diff);
          out[i] = pack2(g);
        }
      }
      if (drow) st_stream16(drow + 8 * v, make_uint4(out[0], out[1], out[2], out[3]));
    };
    if (TOPK) {  // zeros outside the support's vectors, then the candidates densely
      if (drow)
        for (int v = tid; v < nvec; v += kThr)
          if (int(vbin[v]) < tbin) st_stream16(drow + 8 * v, make_uint4(0, 0, 0, 0));
      for (int p = tid; p < nc; p += kThr) {
        const int v = cand[p];
        if (int(vbin[v]) >= tbin) pass2_vector(v, true);
      }
    } else {
      for (int v = tid; v < nvec; v += kThr) pass2_vector(v, false);
    }
    const f2 rs2 = sub2(mk2(0.0f, 0.0f), add2(q2, fs2));

    // this slice's loss sums go to the workspace; the mean kernel adds the
    // slices of each position in rank order (no exchange needed here)
    {
      float f = __fadd_rn(lo2(fs2), hi2(fs2)), r = __fadd_rn(lo2(rs2), hi2(rs2));
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) {
        f = __fadd_rn(f, __shfl_xor_sync(0xFFFFFFFFu, f, d));
        r = __fadd_rn(r, __shfl_xor_sync(0xFFFFFFFFu, r, d));
      }
      if (lane == 0) {
        sh->red[tid >> 5][0] = f;
        sh->red[tid >> 5][1] = r;
      }
    }
    if (TOPK && a.topk_idx) {  // the support in ascending vocabulary order
      int32_t* out = a.topk_idx + row * a.K + sel_before;
      const int32_t vb = int32_t(v0);
      const int room = a.K - sel_before;  // a support larger than K is never written past the row
      ordered_scan(
          tsl, cand, nc, selected,
          [&](int i, int pos) {
            if (pos < room) out[pos] = vb + i;
          },
          sh);
    }
    __syncthreads();  // every read of this row's buffer and histograms is done
    if (tid == 0) {
      float F = 0.0f, R = 0.0f;
      for (int k = 0; k < kWarps; ++k) {
        F = __fadd_rn(F, sh->red[k][0]);
        R = __fadd_rn(R, sh->red[k][1]);
      }
      a.part[(row * kCl + rank) * 2] = F;
      a.part[(row * kCl + rank) * 2 + 1] = R;
      if (rank == 0) {
        a.rowx[2 * row] = conf;
        a.rowx[2 * row + 1] = SE;
      }
      if (tnext < (unsigned long long)nval) {  // the buffer is free: refill it
        sm100::fence_proxy_async_smem();
        prefetch(a.rows[tnext], 0);
      }
    }
    if (TOPK) {  // peers read these before the support-statistics exchange
      for (int i = tid; i < 2 * kHistWords; i += kThr) vhist[i] = 0;
      if (tid < 16) tk->hist2[tid] = 0;
    }
    __syncthreads();
    tcur = tnext;
  }
  // ignored positions: zero gradient slices (and -1 support indices); no
  // exchange, so the (position, slice) pairs are spread over every CTA
  {
    const int64_t first = nval, npair = (a.T - first) * kCl;
    for (int64_t p = blockIdx.x; p < npair; p += int64_t(gridDim.x)) {
      const int64_t row = a.rows[first + p / kCl];
      const int64_t vr0 = (p % kCl) * int64_t(a.S);
      int64_t n = a.V - vr0;
      if (n > a.S) n = a.S;
      if (n < 0) n = 0;
      if (a.ds)
        for (int v = tid; v < int(n >> 3); v += kThr)
          st_stream16(a.ds + row * a.V + vr0 + 8 * v, make_uint4(0, 0, 0, 0));
      if (TOPK && p % kCl == 0 && a.topk_idx)
        for (int j = tid; j < a.K; j += kThr) a.topk_idx[row * a.K + j] = -1;
    }
  }
  // a copy whose wait timed out may still be landing: give it time before exit
  if (tid == 0 && sh->err) {
    wait_phase(&sh->full[0], (uses[0] + 1u) & 1u);
    wait_phase(&sh->full[1], (uses[1] + 1u) & 1u);
    atomicExch(&a.ws_head[1], 1);
  }
  // no CTA leaves while a peer may still read its shared memory
  cluster_sync();
}

// ---------------------------------------------------------------------------
// Top-K loss, one CTA per position
// ---------------------------------------------------------------------------
// The top-K loss and its gradient depend on the student only at the teacher's
// K largest logits, so a position needs one read of the teacher row, the
// student's values on the support and the gradient row (zeros outside the
// support).  One CTA takes a whole position, with block barriers only:
//   pass 1   the teacher row streamed once: the whole-vocabulary statistics
//            (conf), the largest key, and the 12-bit bin of every 8-element
//            vector maximum with their histogram (kept in shared memory)
//   bound    the K-th largest vector maximum's bin bounds the K-th element
//   exact    the elements of the candidate vectors (maximum at or above the
//            bound, re-read, from L2) counted by key: exact 16-bit keys when
//            they span at most 4096 of them, else 12-bit bins and then the
//            low 4 bits of the threshold bin; the walk gives the threshold key
//   ties     elements equal to it are taken in index order (each thread owns
//            a contiguous range of vectors; one block scan)
//   support  statistics of both distributions over the support, with the
//            student's support vectors gathered from device memory
//   pass 2   the gradient row: zeros outside the candidate vectors, the
//            masked gradient in them; the loss sums
// Positions are handed out by ticket as in kd_loss_kernel; the row's sums go
// to slot 0 of the workspace's per-slice sums (the other slots hold zeros).
template <bool RGRAD>
__global__ void __launch_bounds__(kThr, kMinBlocks) kd_topk_row_kernel(const KdArgs a) {
  extern __shared__ __align__(16) uint8_t kd_smem[];
  KdShared* sh = reinterpret_cast<KdShared*>(kd_smem);
  uint32_t* vhist = reinterpret_cast<uint32_t*>(kd_smem + sizeof(KdShared));  // [4096] vector-max bins
  uint32_t* hist1 = vhist + kHist1;                                            // [4096] element bins
  uint32_t* hist2 = hist1 + kHist1;                                            // [16] low nibbles
  uint16_t* vbin = reinterpret_cast<uint16_t*>(hist2 + 16);                    // [nvec] vector bins
  constexpr int kHistAll = 2 * kHist1 + 16;
  const int tid = threadIdx.x, lane = tid & 31;
  const int nvec = int(a.V >> 3);  // V % 8 == 0
  const int vbin_bytes = (2 * nvec + 15) / 16 * 16;  // the bin array (16-byte multiple)
  const int per = (nvec + kThr - 1) / kThr;  // this thread's contiguous vectors [c0, c1)
  const int c0 = min(nvec, tid * per), c1 = min(nvec, c0 + per);
  const int nval = a.ws_head[0];
  const float ks = a.ks;
  const float gsc = nval > 0 ? a.grad_scale * a.tau / float(nval) : 0.0f;
  for (int i = tid; i < kHistAll; i += kThr) vhist[i] = 0u;
  if (tid == 0) sh->tk = atomicAdd(a.ticket, 1ull);
  __syncthreads();
  unsigned long long tcur = sh->tk;
  __syncthreads();

  while (tcur < (unsigned long long)nval) {
    const int64_t row = a.rows[tcur];
    if (tid == 0) sh->tk = atomicAdd(a.ticket, 1ull);  // the next one, read at the end
    const uint16_t* trow = a.t + row * a.V;
    const uint16_t* srow = a.s + row * a.V;
    uint16_t* drow = a.ds ? a.ds + row * a.V : nullptr;
    const int64_t lab = a.labels[row];  // in [0, V): a valid position

    // ---- pass 1: the teacher row ----------------------------------------------
    float tmax = -INFINITY, xl = 0.0f;
    f2 zt = 0;
    {
      const f2 KS = mk2(ks, ks);
      for (int v0 = tid; v0 < nvec; v0 += 4 * kThr) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + u * kThr;
          w[u] = v < nvec ? ld_row16(trow + 8 * int64_t(v)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + u * kThr;
          if (v >= nvec) continue;
          const float vt = vmax8(w[u]);
          const uint32_t kb = key_of_f(vt) >> 4;
          vbin[v] = uint16_t(kb);
          atomicAdd(&vhist[kb], 1u);
          if (vt > tmax) {
            const float f = ex2(__fmul_rn(__fsub_rn(tmax, vt), ks));
            zt = mul2(zt, mk2(f, f));
            tmax = vt;
          }
          const f2 TM = mk2(tmax, tmax);
#pragma unroll
          for (int i = 0; i < 4; ++i) zt = add2(zt, ex2x2(mul2(sub2(bf2(word(w[u], i)), TM), KS)));
          if ((lab >> 3) == v) {  // the label's teacher logit
            const int j = int(lab & 7);
            xl = __uint_as_float(((word(w[u], j >> 1) >> ((j & 1) * 16)) & 0xFFFFu) << 16);
          }
        }
      }
    }
    const Rec R1 = block_rec<true>(
        warp_rec<true>(Rec{Online{tmax, __fadd_rn(lo2(zt), hi2(zt)), 0.0f}, online_empty(), 0.0f, xl,
                           tmax > -INFINITY ? int(key_of_f(tmax)) : 0},
                       ks),
        sh, ks);
    const Online T_ = R1.t;
    const float conf = ex2(__fmaf_rn(__fsub_rn(R1.v, T_.m), ks, -log2f(T_.z)));
    const int top = R1.k >> 4;

    // ---- candidate vectors -------------------------------------------------------
    int b0 = 0, above = 0;
    if (!find_local(vhist, top, a.K, b0, above, sh)) b0 = 0;  // fewer than K vectors: all
    // the vectors whose maximum is at or above the bound, ascending, written
    // over the bins: each thread marks its range (at most 256 vectors) in a
    // register mask before any thread writes
    uint16_t* cand = vbin;
    int nc;
    {
      uint32_t msk[kMaxPer / 32];
      int cc = 0;
#pragma unroll
      for (int q = 0; q < kMaxPer / 32; ++q) {
        uint32_t bits = 0;
        const int n = min(32, (c1 - c0) - 32 * q);
        for (int j = 0; j < n; ++j) bits |= (int(vbin[c0 + 32 * q + j]) >= b0 ? 1u : 0u) << j;
        msk[q] = bits;
        cc += __popc(bits);
      }
      int total;
      int pos = block_scan(cc, total, sh) - cc;  // its barriers end every read of the bins
#pragma unroll
      for (int q = 0; q < kMaxPer / 32; ++q)
        for (uint32_t bits = msk[q]; bits; bits &= bits - 1)
          cand[pos++] = uint16_t(c0 + 32 * q + __ffs(bits) - 1);
      nc = total;
      __syncthreads();
    }
    // The candidates' teacher vectors are read from device memory once (the
    // row has usually left L2 by now) and kept in the rest of the bin array,
    // as many as fit; the later steps read them there.
    uint4* tstage = reinterpret_cast<uint4*>(vbin) + (2 * nc + 15) / 16;
    const int tcap = int((uint4*)(reinterpret_cast<uint8_t*>(vbin) + vbin_bytes) - tstage);
    auto tvec = [&](int p, int v) {
      return p < tcap ? tstage[p] : ld_row16(trow + 8 * int64_t(v));
    };
    // The student vectors of the first kPcap candidates are fetched along
    // with them and kept in the vector-max histogram (free now); those of
    // later candidates that hold support are fetched by the statistics and
    // kept in the element histogram (free by then) for pass 2.
    uint4* pstage = reinterpret_cast<uint4*>(vhist);
    constexpr int kPcap = kHist1 * 4 / 16;
    // Candidate vectors are visited strided (every lane busy), four per
    // thread in flight: for_cand(f) calls f(v, w) for each candidate v with w
    // its teacher vector (from device memory, staged on the way).
    auto for_cand = [&](auto&& f) {
      for (int p0 = tid; p0 < nc; p0 += 4 * kThr) {
        uint4 w[4];
        int v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int p = p0 + u * kThr;
          v[u] = p < nc ? int(cand[p]) : -1;
          w[u] = v[u] >= 0 ? ld_row16(trow + 8 * int64_t(v[u])) : make_uint4(0, 0, 0, 0);
          if (v[u] >= 0 && p < kPcap) pstage[p] = ld_row16(srow + 8 * int64_t(v[u]));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (v[u] >= 0) {
            const int p = p0 + u * kThr;
            if (p < tcap) tstage[p] = w[u];
            f(v[u], w[u]);
          }
      }
    };

    // ---- threshold key -----------------------------------------------------------
    const bool exact = (top - b0 + 1) * 16 <= kHist1;
    const uint32_t kbase = uint32_t(b0) << 4;
    for_cand([&](int, const uint4& w) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t k = key_of(w, j);
        if (int(k >> 4) >= b0) atomicAdd(&hist1[exact ? k - kbase : (k >> 4)], 1u);
      }
    });
    __syncthreads();
    uint32_t tkey;
    int need, eq_total;  // equal keys to take (index order), equal keys present
    if (exact) {
      int tb = 0;
      find_local(hist1, int(((uint32_t(top) + 1u) << 4) - 1u - kbase), a.K, tb, above, sh);
      tkey = kbase + uint32_t(tb);
      need = a.K - above;
      eq_total = int(hist1[tb]);
    } else {
      int bstar = 0;
      find_local(hist1, top, a.K, bstar, above, sh);
      for (int p = tid; p < nc; p += kThr) {
        const uint4 w = tvec(p, int(cand[p]));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t k = key_of(w, j);
          if (int(k >> 4) == bstar) atomicAdd(&hist2[k & 15u], 1u);
        }
      }
      __syncthreads();
      if (tid == 0) {
        const int q = a.K - above;
        int cum = 0, l = 15;
        for (; l > 0; --l) {
          if (cum + int(hist2[l]) >= q) break;
          cum += int(hist2[l]);
        }
        sh->sel[2] = int((uint32_t(bstar) << 4) | uint32_t(l));
        sh->sel[3] = q - cum;
        sh->sel[4] = int(hist2[l]);
      }
      __syncthreads();
      tkey = uint32_t(sh->sel[2]);
      need = sh->sel[3];
      eq_total = sh->sel[4];
      __syncthreads();
    }
    const int tbin = int(tkey >> 4);
    __syncthreads();  // every read of the histograms is done: the student stage reuses them

    // ---- ties: the first `need` elements equal to the key, in index order ----
    int idx_lim = 8 * nvec;  // every equal element taken
    if (eq_total > need) {
      if (tid == 0) sh->sel[5] = -1;
      int base = 0;  // the same in every thread
      for (int p0 = 0; p0 < nc && base < need; p0 += kThr) {
        const int p = p0 + tid;
        uint32_t em = 0;
        int v = 0;
        if (p < nc) {
          v = cand[p];
          const uint4 w = tvec(p, v);
#pragma unroll
          for (int j = 0; j < 8; ++j) em |= (key_of(w, j) == tkey ? 1u : 0u) << j;
        }
        const int e = __popc(em);
        int tot;
        const int before = base + block_scan(e, tot, sh) - e;
        if (before < need && before + e >= need) {  // the need-th is in this vector
          uint32_t bits = em;
          for (int k = before + 1; k < need; ++k) bits &= bits - 1;
          sh->sel[5] = 8 * v + (__ffs(bits) - 1);
        }
        base += tot;
      }
      __syncthreads();
      idx_lim = sh->sel[5];
    }
    auto selected = [&](int i, uint32_t k) { return k > tkey || (k == tkey && i <= idx_lim); };
    // candidate vectors holding support elements: their maximum's bin reaches tbin
    auto holds_support = [&](const uint4& w) { return int(key_of_f(vmax8(w)) >> 4) >= tbin; };

    // ---- statistics over the support ---------------------------------------------
    // each distribution as (raw maximum M, L = log2 of the sum of 2^((v - M) ks))
    uint4* sstage = reinterpret_cast<uint4*>(hist1) - kPcap;  // candidates kPcap ..
    constexpr int kScap = kHist1 * 4 / 16;
    Online ut = online_empty(), us = online_empty();
    int cnt = 0;
    for (int p0 = tid; p0 < nc; p0 += 4 * kThr) {
      uint4 w[4], x[4];
      int v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int p = p0 + u * kThr;
        v[u] = p < nc ? int(cand[p]) : -1;
        w[u] = v[u] >= 0 ? tvec(p, v[u]) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int p = p0 + u * kThr;
        if (v[u] >= 0 && !holds_support(w[u])) v[u] = -1;
        x[u] = v[u] < 0     ? make_uint4(0, 0, 0, 0)
               : p < kPcap ? pstage[p]
                           : ld_row16(srow + 8 * int64_t(v[u]));
        if (v[u] >= 0 && p >= kPcap && p < kPcap + kScap) sstage[p] = x[u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (v[u] < 0) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (!selected(8 * v[u] + j, key_of(w[u], j))) continue;
          const uint32_t tw = word(w[u], j >> 1), sw = word(x[u], j >> 1);
          const float t = __uint_as_float(j & 1 ? tw & 0xFFFF0000u : tw << 16);
          const float sv = __uint_as_float(j & 1 ? sw & 0xFFFF0000u : sw << 16);
          ut = online_merge(ut, Online{t, 1.0f, 0.0f}, ks);
          us = online_merge(us, Online{sv, 1.0f, __fmul_rn(__fsub_rn(sv, t), ks)}, ks);
          ++cnt;
        }
      }
    }
    const Rec RS = block_rec<false>(warp_rec<false>(Rec{ut, us, 0.0f, 0.0f, cnt}, ks), sh, ks);
    const float m_t = RS.t.m, m_s = RS.s.m, l_t = log2f(RS.t.z), l_s = log2f(RS.s.z);
    const float bz = RS.s.b / RS.s.z;

    // ---- pass 2: the gradient row and the loss sums ----------------------------
    // zeros everywhere first; after a barrier the support's vectors over them
    if (drow)
      for (int v = tid; v < nvec; v += kThr)
        st_stream16(drow + 8 * int64_t(v), make_uint4(0, 0, 0, 0));
    __syncthreads();
    const float dl = __fmaf_rn(__fsub_rn(m_t, m_s), ks, __fsub_rn(l_t, l_s));
    const float rkl0 = kLn2 * (bz + dl);
    const float wf = a.type == AQFQ_KD_KL ? 1.0f : a.type == AQFQ_KD_RKL ? 0.0f : 1.0f - conf;
    const float wr2 = a.type == AQFQ_KD_KL ? 0.0f : a.type == AQFQ_KD_RKL ? 1.0f : conf;
    const f2 KS = mk2(ks, ks), NLT = mk2(-l_t, -l_t), NLS = mk2(-l_s, -l_s);
    const f2 MT = mk2(m_t, m_t), MS = mk2(m_s, m_s);
    const float kl = ks * kLn2, ndl = -dl * kLn2;
    const f2 KL2 = mk2(kl, kl), NDL = mk2(ndl, ndl);
    const f2 WF = mk2(gsc * wf, gsc * wf), NWF = mk2(-gsc * wf, -gsc * wf);
    const f2 NWR = mk2(-gsc * wr2, -gsc * wr2);
    const float c = gsc * wf - gsc * wr2 * rkl0;
    const f2 C2 = mk2(c, c);
    f2 fs2 = 0, q2 = 0;
    for (int p0 = tid; p0 < nc; p0 += 4 * kThr) {
      uint4 w[4], x[4];
      int v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int p = p0 + u * kThr;
        v[u] = p < nc ? int(cand[p]) : -1;
        w[u] = v[u] >= 0 ? tvec(p, v[u]) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int p = p0 + u * kThr;
        if (v[u] >= 0 && !holds_support(w[u])) v[u] = -1;
        x[u] = v[u] < 0                 ? make_uint4(0, 0, 0, 0)
               : p < kPcap             ? pstage[p]
               : p < kPcap + kScap     ? sstage[p]
                                       : ld_row16(srow + 8 * int64_t(v[u]));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (v[u] < 0) continue;
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const f2 t2 = bf2(word(w[u], i)), s2 = bf2(word(x[u], i));
          f2 pt = ex2x2(fma2(sub2(t2, MT), KS, NLT)), ps = ex2x2(fma2(sub2(s2, MS), KS, NLS));
          const bool in0 = selected(8 * v[u] + 2 * i, key_of(w[u], 2 * i));
          const bool in1 = selected(8 * v[u] + 2 * i + 1, key_of(w[u], 2 * i + 1));
          pt = mk2(in0 ? lo2(pt) : 0.0f, in1 ? hi2(pt) : 0.0f);
          ps = mk2(in0 ? lo2(ps) : 0.0f, in1 ? hi2(ps) : 0.0f);
          const f2 dn = fma2(sub2(t2, s2), KL2, NDL);  // log p_t - log p_s in nats
          const f2 diff = sub2(ps, pt);
          fs2 = add2(fs2, fma2(pt, dn, diff));
          q2 = fma2(diff, dn, q2);
          const f2 g = RGRAD ? fma2(ps, fma2(NWR, dn, C2), mul2(NWF, pt)) : mul2(WF, diff);
          out[i] = pack2(g);
        }
        if (drow) st_stream16(drow + 8 * int64_t(v[u]), make_uint4(out[0], out[1], out[2], out[3]));
      }
    }
    const f2 rs2 = sub2(mk2(0.0f, 0.0f), add2(q2, fs2));
    {
      float f = __fadd_rn(lo2(fs2), hi2(fs2)), r = __fadd_rn(lo2(rs2), hi2(rs2));
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) {
        f = __fadd_rn(f, __shfl_xor_sync(0xFFFFFFFFu, f, d));
        r = __fadd_rn(r, __shfl_xor_sync(0xFFFFFFFFu, r, d));
      }
      if (lane == 0) {
        sh->red[tid >> 5][0] = f;
        sh->red[tid >> 5][1] = r;
      }
    }
    if (a.topk_idx) {  // the support in ascending vocabulary order (candidates are)
      int32_t* out = a.topk_idx + row * a.K;
      int base = 0;  // the same in every thread
      for (int p0 = 0; p0 < nc; p0 += kThr) {
        const int p = p0 + tid;
        uint32_t sm8 = 0;
        int v = 0;
        if (p < nc) {
          v = cand[p];
          const uint4 w = tvec(p, v);
#pragma unroll
          for (int j = 0; j < 8; ++j) sm8 |= (selected(8 * v + j, key_of(w, j)) ? 1u : 0u) << j;
        }
        const int e = __popc(sm8);
        int tot;
        int pos = base + block_scan(e, tot, sh) - e;
        for (uint32_t bits = sm8; bits; bits &= bits - 1) {
          if (pos < a.K) out[pos] = 8 * v + __ffs(bits) - 1;
          ++pos;
        }
        base += tot;
      }
    }
    __syncthreads();  // every read of this row's candidates and sums is done
    if (tid == 0) {
      float F = 0.0f, R = 0.0f;
      for (int k = 0; k < kWarps; ++k) {
        F = __fadd_rn(F, sh->red[k][0]);
        R = __fadd_rn(R, sh->red[k][1]);
      }
      a.part[row * kCl * 2] = F;
      a.part[row * kCl * 2 + 1] = R;
      a.rowx[2 * row] = conf;
      a.rowx[2 * row + 1] = 0.0f;
    }
    if (tid >= 2 && tid < 2 * kCl) a.part[row * kCl * 2 + tid] = 0.0f;  // the other slots
    for (int i = tid; i < kHistAll; i += kThr) vhist[i] = 0u;
    const unsigned long long tnext = sh->tk;
    __syncthreads();
    tcur = tnext;
  }
  // ignored positions: zero gradient rows (and -1 support indices)
  for (int64_t p = blockIdx.x; p < a.T - nval; p += int64_t(gridDim.x)) {
    const int64_t row = a.rows[nval + p];
    if (a.ds)
      for (int v = tid; v < nvec; v += kThr)
        st_stream16(a.ds + row * a.V + 8 * int64_t(v), make_uint4(0, 0, 0, 0));
    if (a.topk_idx)
      for (int j = tid; j < a.K; j += kThr) a.topk_idx[row * a.K + j] = -1;
  }
}

// Number of positions whose label lies in [0, V) (head[0]) and the list of
// positions (rows): the valid ones ascending at [0, head[0]), the ignored ones
// after them (filled from the end of the list); clears the error word, the
// mean kernel's ticket and the loss kernel's position ticket.  One block, in
// chunks of 4 rows per thread: one scan counts valid (low 16 bits) and
// ignored (high 16 bits) rows together.
__global__ void kd_count_kernel(const int32_t* labels, int64_t T, int64_t V, int32_t* head,
                                int64_t* rows) {
  __shared__ int part[32];
  __shared__ int64_t base_v, base_i;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = int(blockDim.x >> 5);
  if (threadIdx.x == 0) {
    base_v = 0;
    base_i = 0;
  }
  __syncthreads();
  for (int64_t c0 = 0; c0 < T; c0 += int64_t(blockDim.x) * 4) {
    const int64_t i0 = c0 + int64_t(threadIdx.x) * 4;
    uint32_t fv = 0, fi = 0;  // bit j: row i0 + j valid / ignored
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i0 + j < T) {
        const int32_t l = labels[i0 + j];
        if (l >= 0 && int64_t(l) < V) fv |= 1u << j;
        else fi |= 1u << j;
      }
    const int packed = __popc(fv) | (__popc(fi) << 16);  // a chunk has at most 4096 rows
    int x = packed;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) part[w] = x;
    __syncthreads();
    int before = 0, total = 0;
    for (int k = 0; k < nw; ++k) {
      if (k < w) before += part[k];
      total += part[k];
    }
    const int ex = x - packed + before;
    int64_t pv = base_v + (ex & 0xFFFF), pi = base_i + (ex >> 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((fv >> j) & 1u) rows[pv++] = i0 + j;
      else if ((fi >> j) & 1u) rows[T - 1 - pi++] = i0 + j;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      base_v += total & 0xFFFF;
      base_i += total >> 16;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    head[0] = int(base_v);
    head[1] = 0;
    head[2] = 0;  // the mean kernel's ticket
    *reinterpret_cast<unsigned long long*>(head + 4) = 0ull;  // the loss kernel's position ticket
  }
}

// Per position: forward / reverse KL = tau^2 x the sum of the slices' sums
// (rank order), the loss of the selected type, written to token_loss; then
// losses[k] = the sums over the valid positions / their number (double
// accumulation in a fixed order: block b sums positions [b c, b c + c) by a
// fixed pattern, the last block to finish adds the blocks' sums in block
// order); NaN if a copy wait of the loss kernel timed out.
constexpr int kMeanBlocks = 32;
__global__ void __launch_bounds__(256) kd_mean_kernel(const float* part, const float* rowx,
                                                      const int32_t* labels, int32_t* head,
                                                      double* bsum, int64_t T, int64_t V,
                                                      int type, float tau2, float* token_loss,
                                                      float* losses) {
  __shared__ double acc[8][3];
  __shared__ int last;
  const int64_t c = (T + gridDim.x - 1) / gridDim.x;
  const int64_t i0 = int64_t(blockIdx.x) * c;
  const int64_t i1 = i0 + c < T ? i0 + c : T;
  double s[3] = {0.0, 0.0, 0.0};
  for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const int32_t l = labels[i];
    float loss = 0.0f;
    if (l >= 0 && int64_t(l) < V) {
      float F = 0.0f, R = 0.0f;
      for (int r = 0; r < kCl; ++r) {
        F = __fadd_rn(F, part[(i * kCl + r) * 2]);
        R = __fadd_rn(R, part[(i * kCl + r) * 2 + 1]);
      }
      F = tau2 * F;
      R = tau2 * R;
      const float conf = rowx[2 * i];
      loss = type == AQFQ_KD_MSE   ? rowx[2 * i + 1] / float(V)
             : type == AQFQ_KD_KL  ? F
             : type == AQFQ_KD_RKL ? R
                                   : conf * R + (1.0f - conf) * F;
      s[0] += double(loss);
      s[1] += double(F);
      s[2] += double(R);
    }
    if (token_loss) token_loss[i] = loss;
  }
#pragma unroll
  for (int k = 0; k < 3; ++k)
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) s[k] += __shfl_xor_sync(0xFFFFFFFFu, s[k], d);
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int k = 0; k < 3; ++k) acc[threadIdx.x >> 5][k] = s[k];
  __syncthreads();
  if (threadIdx.x < 3) {
    double t = 0.0;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) t += acc[w][threadIdx.x];
    bsum[blockIdx.x * 3 + threadIdx.x] = t;
    __threadfence();  // each writer's sum is visible device-wide before the ticket
  }
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&head[2], 1) == int(gridDim.x) - 1;
  __syncthreads();
  if (last && threadIdx.x < 3) {
    __threadfence();
    double t = 0.0;
    for (int b = 0; b < int(gridDim.x); ++b)
      t += *reinterpret_cast<volatile const double*>(&bsum[b * 3 + threadIdx.x]);
    const int n = T > 0 ? head[0] : 0;
    float r = n > 0 ? float(t / double(n)) : 0.0f;
    if (T > 0 && head[1] != 0) r = __int_as_float(0x7FC00000);
    losses[threadIdx.x] = r;
  }
}

}  // namespace
}  // namespace aqfq

// ---- host side -------------------------------------------------------------

namespace {

using namespace aqfq;

// workspace: [0, 256) int32 valid count, error word and the mean kernel's
// ticket, at byte 16 the 64-bit position ticket; [256, 1024) the mean
// kernel's per-block double sums; then part [T, kCl, 2] and rowx [T, 2]
// floats and the position list [T] int64, each on a 256-byte boundary
constexpr size_t kWsHead = 1024;
constexpr size_t kWsBsum = 256;
static_assert(kWsBsum + kMeanBlocks * 3 * sizeof(double) <= kWsHead, "block sums fit the head");
size_t ws_part_bytes(int64_t T) { return (size_t(T) * kCl * 8 + 255) / 256 * 256; }

size_t kd_smem_bytes(int32_t S, bool topk) {
  const size_t vbin = topk ? size_t((S / 8 + 7) / 8 * 8) * 4 : 0;  // vector bins + candidate list
  // each buffer: the teacher's slice, and the student's but for top-K
  return sizeof(KdShared) + (topk ? size_t(2 * kHistWords) * 4 + sizeof(TopkShared) : 0) + vbin +
         size_t(S) * (topk ? 2 : 4) * kNbuf;
}

int max_smem_optin() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  return v;
}

template <bool TOPK, bool RGRAD, bool MSE>
cudaError_t launch_kd(const KdArgs& a, size_t smem, cudaStream_t st) {
  auto kern = kd_loss_kernel<TOPK, RGRAD, MSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  // all of the unified L1 / shared memory as shared memory: two CTAs per SM
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThr);
  cfg.gridDim = dim3(kCl);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  if (int64_t(clusters) > a.T) clusters = int(a.T);
  cfg.gridDim = dim3(unsigned(clusters * kCl));
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// the top-K row kernel: bookkeeping, two 4096-bin histograms and the low
// nibbles (32-bit counters), and the bin of every 8-element vector of a row
size_t kd_row_smem_bytes(int64_t V) {
  return sizeof(KdShared) + size_t(2 * kHist1 + 16) * 4 + (size_t(V / 8) * 2 + 15) / 16 * 16;
}

template <bool RGRAD>
cudaError_t launch_kd_row(const KdArgs& a, size_t smem, cudaStream_t st) {
  auto kern = kd_topk_row_kernel<RGRAD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThr, smem);
  if (e != cudaSuccess) return e;
  const int sms = aqfq::sm_count();
  if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
  int64_t blocks = int64_t(per_sm) * sms;  // one wave, persistent over positions
  if (blocks > a.T) blocks = a.T;
  kern<<<unsigned(blocks), kThr, smem, st>>>(a);
  return cudaGetLastError();
}

bool al(const void* p, uintptr_t b) { return (reinterpret_cast<uintptr_t>(p) & (b - 1)) == 0; }

}  // namespace

extern "C" size_t aqfq_kd_workspace_bytes(int64_t T) {
  if (T < 0) return 0;
  return kWsHead + ws_part_bytes(T) + 2 * ((size_t(T) * 8 + 255) / 256 * 256);
}

extern "C" aqfq_status aqfq_kd_loss(int kd_type, const void* student, const void* teacher,
                                    const int32_t* labels, int64_t T, int64_t V, int32_t topk,
                                    float temperature, float grad_scale, float* losses,
                                    float* token_loss, void* dstudent, int32_t* topk_idx,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (kd_type < AQFQ_KD_KL || kd_type > AQFQ_KD_MSE) return AQFQ_ERR_UNSUPPORTED;
  if (T < 0 || V < 8 || V % 8 != 0 || V > 0x7FFFFFF8LL || topk < 0 || int64_t(topk) > V)
    return AQFQ_ERR_SHAPE;
  if (T > (int64_t(1) << 62) / V) return AQFQ_ERR_SHAPE;
  if (!(temperature > 0.0f) || !(temperature < INFINITY) || !(grad_scale == grad_scale))
    return AQFQ_ERR_SHAPE;
  if (kd_type == AQFQ_KD_MSE && (topk != 0 || temperature != 1.0f)) return AQFQ_ERR_UNSUPPORTED;
  if (topk_idx && topk == 0) return AQFQ_ERR_UNSUPPORTED;
  const int32_t S = int32_t(((V + kCl - 1) / kCl + 7) / 8 * 8);
  const bool use_topk = topk > 0;  // K = V takes the top-K path too (it selects everything)
  if (!losses) return AQFQ_ERR_NULL;
  if (T > 0 && (!student || !teacher || !labels)) return AQFQ_ERR_NULL;
  if (!workspace || workspace_bytes < aqfq_kd_workspace_bytes(T)) return AQFQ_ERR_WORKSPACE;
  if (!al(student, 16) || !al(teacher, 16) || !al(dstudent, 16) || !al(labels, 4) ||
      !al(losses, 4) || !al(token_loss, 4) || !al(topk_idx, 4) || !al(workspace, 16))
    return AQFQ_ERR_ALIGN;
  const size_t smem = kd_smem_bytes(S, use_topk);
  const int optin = max_smem_optin();
  if (optin <= 0) return AQFQ_ERR_CUDA;
  // top-K: one CTA per position where its layout fits, else the cluster kernel
  const size_t row_smem = kd_row_smem_bytes(V);
  const bool row_path = use_topk && kd_type != AQFQ_KD_MSE && row_smem <= size_t(optin) &&
                        V / 8 <= int64_t(kThr) * kMaxPer;
  if (!row_path && smem > size_t(optin)) return AQFQ_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* head = static_cast<int32_t*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kWsHead);
  float* rowx = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kWsHead + ws_part_bytes(T));
  int64_t* rows = reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(rowx) + (size_t(T) * 8 + 255) / 256 * 256);
  kd_count_kernel<<<1, 1024, 0, st>>>(labels, T, V, head, rows);
  if (cudaGetLastError() != cudaSuccess) return AQFQ_ERR_CUDA;
  if (T > 0) {
    KdArgs a;
    a.s = static_cast<const uint16_t*>(student);
    a.t = static_cast<const uint16_t*>(teacher);
    a.labels = labels;
    a.ws_head = head;
    a.rows = rows;
    a.ticket = reinterpret_cast<unsigned long long*>(head + 4);
    a.part = part;
    a.rowx = rowx;
    a.ds = static_cast<uint16_t*>(dstudent);
    a.topk_idx = topk_idx;
    a.T = T;
    a.V = V;
    a.S = S;
    a.K = use_topk ? topk : 0;
    a.type = kd_type;
    a.tau = temperature;
    a.tau2 = temperature * temperature;
    a.ks = kLog2e / temperature;
    a.grad_scale = grad_scale;
    const bool rgrad = dstudent && (kd_type == AQFQ_KD_RKL || kd_type == AQFQ_KD_CAKLD);
    cudaError_t e;
    if (kd_type == AQFQ_KD_MSE) e = launch_kd<false, false, true>(a, smem, st);
    else if (row_path) e = rgrad ? launch_kd_row<true>(a, row_smem, st)
                                 : launch_kd_row<false>(a, row_smem, st);
    else if (use_topk) e = rgrad ? launch_kd<true, true, false>(a, smem, st)
                                 : launch_kd<true, false, false>(a, smem, st);
    else e = rgrad ? launch_kd<false, true, false>(a, smem, st)
                   : launch_kd<false, false, false>(a, smem, st);
    if (e != cudaSuccess) return AQFQ_ERR_CUDA;
  }
  double* bsum = reinterpret_cast<double*>(static_cast<uint8_t*>(workspace) + kWsBsum);
  kd_mean_kernel<<<kMeanBlocks, 256, 0, st>>>(part, rowx, labels, head, bsum, T, V, kd_type,
                                              temperature * temperature, token_loss, losses);
  return cudaGetLastError() == cudaSuccess ? AQFQ_OK : AQFQ_ERR_CUDA;
}
