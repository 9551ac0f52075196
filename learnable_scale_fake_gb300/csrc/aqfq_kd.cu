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
// Layout of the work: one cluster of 8 CTAs per position.  CTA r holds the
// vocabulary slice [r S, r S + S) of both rows in shared memory (loaded once
// from HBM), so every later pass reads shared memory and HBM sees each logit
// once and each gradient element once.  Row statistics (max and sum of
// exponentials per row, the top-K histograms, the loss sums) are combined
// across the cluster through distributed shared memory, always in rank
// order, so every CTA holds bit-identical row values and results are
// reproducible.
//
// Numerics: logits are scaled to base-2 units (x = v * log2(e) / tau) and
// exponentials use ex2.approx; log-sum-exp uses the row maximum.  The loss
// is summed per element as p_t d - p_t + p_s (forward) and -p_s d - p_s + p_t
// (reverse), d = log p_t - log p_s in nats: the added -p_t + p_s terms sum to
// zero exactly in real arithmetic and make the sum insensitive, to first
// order, to the rounding of the two normalisers.
#include <cuda_runtime.h>

#include <cstdint>

#include "aqfq.h"
#include "aqfq_internal.h"

namespace aqfq {
namespace {

constexpr int kCl = 8;          // CTAs per position (vocabulary slices)
constexpr int kThr = 512;       // threads per CTA
constexpr int kWarps = kThr / 32;
constexpr int kHist1 = 4096;    // bins: the top 12 bits of the 16-bit teacher key
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

struct KdArgs {
  const uint16_t* s;        // student [T, V] BF16
  const uint16_t* t;        // teacher [T, V] BF16
  const int32_t* labels;    // [T]
  const int32_t* nvalid;    // device: number of valid positions
  float* tok;               // workspace [T, 3]: loss, tau^2 fkl, tau^2 rkl
  float* token_loss;        // optional [T]
  uint16_t* ds;             // optional [T, V] BF16
  int32_t* topk_idx;        // optional [T, K]
  int64_t T, V;
  int32_t S;                // slice length, a multiple of 8
  int32_t K;                // 0: whole vocabulary
  int32_t type;             // AQFQ_KD_*
  float ks;                 // log2(e) / tau
  float tau, tau2, grad_scale;
};

struct __align__(16) KdShared {
  float xbuf[2][16];        // scalar exchanges (alternating)
  float red[kWarps][8];     // block reductions
  int32_t ired[kWarps + 1];
  uint32_t hist2[16];       // low nibble of the keys in the threshold bin
  uint32_t h2all[kCl][16];  // hist2 of every rank
  float label_x;            // teacher x at the label (owner CTA)
  int32_t sel[8];           // threshold bin, need, key, idx_lim, ...
};

// ---------------------------------------------------------------------------
// cluster primitives (PTX: barrier.cluster, mapa, ld.shared::cluster)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
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
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_remote_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_remote_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_remote_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf16f(uint32_t w, int hi) {
  return __uint_as_float(hi ? (w & 0xFFFF0000u) : (w << 16));
}
__device__ __forceinline__ uint32_t pack2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// order-preserving 16-bit key of a BF16 value; -0 and +0 share a key
__device__ __forceinline__ uint32_t okey(uint32_t b) {
  b &= 0xFFFFu;
  if (b == 0x8000u) b = 0;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// (max, sum of 2^(x - max), weighted sum) of a set; z == 0 marks an empty set.
struct Online {
  float m, z, b;
};
__device__ __forceinline__ Online online_empty() { return Online{-INFINITY, 0.0f, 0.0f}; }
// symmetric in its operands (bit for bit), so butterfly lanes agree
__device__ __forceinline__ Online online_merge(Online a, Online c) {
  const float m = fmaxf(a.m, c.m);
  const float fa = a.z != 0.0f ? ex2(a.m - m) : 0.0f;
  const float fc = c.z != 0.0f ? ex2(c.m - m) : 0.0f;
  return Online{m, __fadd_rn(__fmul_rn(a.z, fa), __fmul_rn(c.z, fc)),
                __fadd_rn(__fmul_rn(a.b, fa), __fmul_rn(c.b, fc))};
}
__device__ __forceinline__ Online online_shfl(Online a, int d) {
  return Online{__shfl_xor_sync(0xFFFFFFFFu, a.m, d), __shfl_xor_sync(0xFFFFFFFFu, a.z, d),
                __shfl_xor_sync(0xFFFFFFFFu, a.b, d)};
}
__device__ __forceinline__ Online warp_online(Online a) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) a = online_merge(a, online_shfl(a, d));
  return a;
}

// Block reduction of N sums: every thread gets the totals (fixed order).
template <int N>
__device__ __forceinline__ void block_sum(float (&v)[N], KdShared* sh) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < N; ++i)
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v[i] = __fadd_rn(v[i], __shfl_xor_sync(0xFFFFFFFFu, v[i], d));
  if (l == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) sh->red[w][i] = v[i];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float s = 0.0f;
    for (int k = 0; k < kWarps; ++k) s = __fadd_rn(s, sh->red[k][i]);
    v[i] = s;
  }
  __syncthreads();
}

// Block reduction of two online states (teacher, student) into totals.
__device__ __forceinline__ void block_online2(Online& a, Online& c, KdShared* sh) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  a = warp_online(a);
  c = warp_online(c);
  if (l == 0) {
    sh->red[w][0] = a.m; sh->red[w][1] = a.z; sh->red[w][2] = a.b;
    sh->red[w][3] = c.m; sh->red[w][4] = c.z; sh->red[w][5] = c.b;
  }
  __syncthreads();
  Online ta = online_empty(), tc = online_empty();
  for (int k = 0; k < kWarps; ++k) {
    ta = online_merge(ta, Online{sh->red[k][0], sh->red[k][1], sh->red[k][2]});
    tc = online_merge(tc, Online{sh->red[k][3], sh->red[k][4], sh->red[k][5]});
  }
  a = ta;
  c = tc;
  __syncthreads();
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

// Exchange n <= 16 floats with the cluster: writes them to this CTA's
// exchange slot `par`, synchronises the cluster and returns every rank's
// values in out[rank][i].  A slot is rewritten two exchanges later, after a
// barrier that every CTA passes only once it has read the slot.
template <int N>
__device__ __forceinline__ void cluster_exchange(const float (&mine)[N], float (&out)[kCl][N],
                                                 KdShared* sh, int& par) {
  if (threadIdx.x == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) sh->xbuf[par][i] = mine[i];
  cluster_sync();
#pragma unroll
  for (int r = 0; r < kCl; ++r) {
    const uint32_t base = remote_addr(&sh->xbuf[par][0], r);
#pragma unroll
    for (int i = 0; i < N; ++i) out[r][i] = ld_remote_f32(base + 4u * i);
  }
  par ^= 1;
}


// Visits the slice in index order and calls emit(local index, position) for
// every element whose teacher key satisfies pred(local index, key); the
// position counts those elements from 0 in index order.  All threads call it.
template <class Pred, class Emit>
__device__ __forceinline__ void ordered_scan(const uint16_t* tsl, int nvec, Pred pred, Emit emit,
                                             KdShared* sh) {
  int base = 0;
  for (int v00 = 0; v00 < nvec; v00 += kThr) {
    const int v = v00 + int(threadIdx.x);
    uint32_t m8 = 0;
    if (v < nvec) {
      const uint4 w = *reinterpret_cast<const uint4*>(tsl + 8 * v);
      const uint32_t tw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (pred(8 * v + j, okey(j & 1 ? tw[j >> 1] >> 16 : tw[j >> 1]))) m8 |= 1u << j;
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

// One cluster per position (persistent over positions).  TOPK: restrict to
// the teacher's top-K support.
template <bool TOPK>
__global__ void __launch_bounds__(kThr, 2) kd_loss_kernel(const KdArgs a) {
  extern __shared__ __align__(16) uint8_t kd_smem[];
  KdShared* sh = reinterpret_cast<KdShared*>(kd_smem);
  uint32_t* hist1 = reinterpret_cast<uint32_t*>(kd_smem + sizeof(KdShared));
  uint16_t* tsl = reinterpret_cast<uint16_t*>(kd_smem + sizeof(KdShared) + (TOPK ? kHist1 * 4 : 0));
  uint16_t* ssl = tsl + a.S;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const int64_t v0 = int64_t(rank) * a.S;  // first vocabulary index of this slice
  int64_t n64 = a.V - v0;
  if (n64 > a.S) n64 = a.S;
  if (n64 < 0) n64 = 0;
  const int nvec = int(n64) >> 3;  // V % 8 == 0 and S % 8 == 0
  const int nval = *a.nvalid;
  const bool mse = a.type == AQFQ_KD_MSE;
  const bool need_b = a.ds != nullptr && (a.type == AQFQ_KD_RKL || a.type == AQFQ_KD_CAKLD);
  const float ks = a.ks;
  // gradient factors: d(tau^2 KL(s / tau)) / ds = tau dKL/db, over the mean
  const float gsc = nval > 0 ? (mse ? a.grad_scale * 2.0f / (float(a.V) * float(nval))
                                    : a.grad_scale * a.tau / float(nval))
                             : 0.0f;
  int par = 0;

  for (int64_t row = cluster_id(); row < a.T; row += cluster_count()) {
    const int32_t label = a.labels[row];
    const bool valid = label >= 0 && int64_t(label) < a.V;
    const uint16_t* trow = a.t + row * a.V + v0;
    const uint16_t* srow = a.s + row * a.V + v0;
    uint16_t* drow = a.ds ? a.ds + row * a.V + v0 : nullptr;
    if (!valid) {  // the same decision in every CTA of the cluster: no exchange
      if (drow)
        for (int v = tid; v < nvec; v += kThr) st_stream16(drow + 8 * v, make_uint4(0, 0, 0, 0));
      if (rank == 0) {
        if (TOPK && a.topk_idx)
          for (int j = tid; j < a.K; j += kThr) a.topk_idx[row * a.K + j] = -1;
        if (tid == 0) {
          a.tok[3 * row] = a.tok[3 * row + 1] = a.tok[3 * row + 2] = 0.0f;
          if (a.token_loss) a.token_loss[row] = 0.0f;
        }
      }
      continue;
    }
    if (TOPK) {  // peers finished reading these before the last exchange of the previous row
      for (int i = tid; i < kHist1; i += kThr) hist1[i] = 0;
      if (tid < 16) sh->hist2[tid] = 0;
      __syncthreads();
    }
    const int64_t lloc = int64_t(label) - v0;  // label's index within the slice

    // ---- pass 1: HBM -> shared memory; whole-vocabulary statistics --------
    Online ot = online_empty(), os = online_empty();
    float se = 0.0f, xl = 0.0f;
    for (int v = tid; v < nvec; v += 2 * kThr) {
      const bool two = v + kThr < nvec;
      const uint4 tw0 = ld_stream16(trow + 8 * v), sw0 = ld_stream16(srow + 8 * v);
      uint4 tw1 = make_uint4(0, 0, 0, 0), sw1 = tw1;
      if (two) {
        tw1 = ld_stream16(trow + 8 * (v + kThr));
        sw1 = ld_stream16(srow + 8 * (v + kThr));
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (u == 1 && !two) break;
        const int vv = v + u * kThr;
        const uint4 tw = u ? tw1 : tw0, sw = u ? sw1 : sw0;
        *reinterpret_cast<uint4*>(tsl + 8 * vv) = tw;
        *reinterpret_cast<uint4*>(ssl + 8 * vv) = sw;
        const uint32_t tv[4] = {tw.x, tw.y, tw.z, tw.w}, sv[4] = {sw.x, sw.y, sw.z, sw.w};
        float xt[8], xs[8], tm = -INFINITY, sm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          xt[j] = __fmul_rn(bf16f(tv[j >> 1], j & 1), ks);
          xs[j] = __fmul_rn(bf16f(sv[j >> 1], j & 1), ks);
          tm = fmaxf(tm, xt[j]);
          sm = fmaxf(sm, xs[j]);
        }
        {
          const float m = fmaxf(ot.m, tm);
          float z = __fmul_rn(ot.z, ex2(ot.m - m));
#pragma unroll
          for (int j = 0; j < 8; ++j) z = __fadd_rn(z, ex2(xt[j] - m));
          ot = Online{m, z, 0.0f};
        }
        if (!TOPK) {
          const float m = fmaxf(os.m, sm);
          const float f = ex2(os.m - m);
          float z = __fmul_rn(os.z, f), b = __fmul_rn(os.b, f);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float e = ex2(xs[j] - m);
            z = __fadd_rn(z, e);
            if (need_b) {  // sum of 2^(x_s - m) (x_s - x_t), the difference formed exactly first
              const float dx = __fmul_rn(__fsub_rn(bf16f(sv[j >> 1], j & 1), bf16f(tv[j >> 1], j & 1)), ks);
              b = __fmaf_rn(e, dx, b);
            }
          }
          os = Online{m, z, b};
          if (mse) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float d = __fsub_rn(bf16f(sv[j >> 1], j & 1), bf16f(tv[j >> 1], j & 1));
              se = __fmaf_rn(d, d, se);
            }
          }
        }
        if (TOPK) {
#pragma unroll
          for (int j = 0; j < 8; ++j) atomicAdd(&hist1[okey(j & 1 ? tv[j >> 1] >> 16 : tv[j >> 1]) >> 4], 1u);
        }
        if (lloc >= 8 * vv && lloc < 8 * vv + 8) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (lloc == 8 * vv + j) xl = xt[j];
        }
      }
    }
    block_online2(ot, os, sh);
    {
      float v2[2] = {se, xl};
      block_sum<2>(v2, sh);
      se = v2[0];
      xl = v2[1];
    }
    Online T_ = online_empty(), S_ = online_empty();
    float SE = 0.0f, XL = 0.0f;
    {
      const float mine[8] = {ot.m, ot.z, ot.b, os.m, os.z, os.b, se, xl};
      float all[kCl][8];
      cluster_exchange<8>(mine, all, sh, par);
#pragma unroll
      for (int r = 0; r < kCl; ++r) {
        T_ = online_merge(T_, Online{all[r][0], all[r][1], all[r][2]});
        S_ = online_merge(S_, Online{all[r][3], all[r][4], all[r][5]});
        SE = __fadd_rn(SE, all[r][6]);
        XL = __fadd_rn(XL, all[r][7]);
      }
    }
    // conf: the whole-vocabulary teacher probability of the label
    const float conf = ex2(XL - (T_.m + log2f(T_.z)));

    // ---- top-K support: threshold key, ties by index ------------------------
    uint32_t tkey = 0;
    int idx_lim = -1;
    if (TOPK) {
      // thread tid owns bins [8 g, 8 g + 8) with g = kThr - 1 - tid, so the
      // scan over threads runs from the largest keys down
      const int g = kThr - 1 - tid;
      uint32_t hb[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int r = 0; r < kCl; ++r) {
        const uint32_t base = remote_addr(hist1 + 8 * g, r);
        const uint4 p = ld_remote_v4(base), q = ld_remote_v4(base + 16);
        hb[0] += p.x; hb[1] += p.y; hb[2] += p.z; hb[3] += p.w;
        hb[4] += q.x; hb[5] += q.y; hb[6] += q.z; hb[7] += q.w;
      }
      int c = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) c += int(hb[j]);
      int total;
      const int incl = block_scan(c, total, sh);
      if (incl - c < a.K && incl >= a.K) {
        int cum = incl - c;
        for (int j = 7; j >= 0; --j) {
          if (cum + int(hb[j]) >= a.K) {
            sh->sel[0] = 8 * g + j;
            sh->sel[1] = a.K - cum;
            break;
          }
          cum += int(hb[j]);
        }
      }
      __syncthreads();
      const uint32_t bstar = uint32_t(sh->sel[0]);
      const int need = sh->sel[1];
      for (int v = tid; v < nvec; v += kThr) {
        const uint4 w = *reinterpret_cast<const uint4*>(tsl + 8 * v);
        const uint32_t tw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t k = okey(j & 1 ? tw[j >> 1] >> 16 : tw[j >> 1]);
          if ((k >> 4) == bstar) atomicAdd(&sh->hist2[k & 15u], 1u);
        }
      }
      __syncthreads();
      cluster_sync();
      if (tid < kCl * 16) sh->h2all[tid >> 4][tid & 15] = ld_remote_u32(remote_addr(&sh->hist2[tid & 15], tid >> 4));
      __syncthreads();
      if (tid == 0) {
        int cum = 0, l = 15;
        for (; l > 0; --l) {
          int h = 0;
          for (int r = 0; r < kCl; ++r) h += int(sh->h2all[r][l]);
          if (cum + h >= need) break;
          cum += h;
        }
        const int q = need - cum;  // elements equal to the threshold key to take
        int before = 0;
        for (uint32_t r = 0; r < rank; ++r) before += int(sh->h2all[r][l]);
        const int eq = int(sh->h2all[rank][l]);
        int take = q - before;
        take = take < 0 ? 0 : (take > eq ? eq : take);
        sh->sel[2] = int((bstar << 4) | uint32_t(l));
        sh->sel[3] = take;
        sh->sel[4] = eq;
        sh->sel[5] = -1;
      }
      __syncthreads();
      tkey = uint32_t(sh->sel[2]);
      const int take = sh->sel[3], eq = sh->sel[4];
      if (take == eq) {
        idx_lim = 8 * nvec;
      } else if (take > 0) {  // the take-th equal element in index order
        ordered_scan(
            tsl, nvec, [&](int, uint32_t k) { return k == tkey; },
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
    float lse_t, lse_s, rkl0;
    int sel_before = 0;
    if (TOPK) {
      Online ut = online_empty(), us = online_empty();
      float cnt = 0.0f;
      for (int v = tid; v < nvec; v += kThr) {
        const uint4 w = *reinterpret_cast<const uint4*>(tsl + 8 * v);
        const uint4 x = *reinterpret_cast<const uint4*>(ssl + 8 * v);
        const uint32_t tw[4] = {w.x, w.y, w.z, w.w}, sw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (!selected(8 * v + j, okey(j & 1 ? tw[j >> 1] >> 16 : tw[j >> 1]))) continue;
          const float t = bf16f(tw[j >> 1], j & 1), s = bf16f(sw[j >> 1], j & 1);
          const float xt = __fmul_rn(t, ks), xs = __fmul_rn(s, ks);
          ut = online_merge(ut, Online{xt, 1.0f, 0.0f});
          const float dx = __fmul_rn(__fsub_rn(s, t), ks);
          us = online_merge(us, Online{xs, 1.0f, dx});
          cnt += 1.0f;
        }
      }
      block_online2(ut, us, sh);
      float c1[1] = {cnt};
      block_sum<1>(c1, sh);
      const float mine[8] = {ut.m, ut.z, ut.b, us.m, us.z, us.b, c1[0], 0.0f};
      float all[kCl][8];
      cluster_exchange<8>(mine, all, sh, par);
      Online UT = online_empty(), US = online_empty();
#pragma unroll
      for (int r = 0; r < kCl; ++r) {
        UT = online_merge(UT, Online{all[r][0], all[r][1], all[r][2]});
        US = online_merge(US, Online{all[r][3], all[r][4], all[r][5]});
        if (uint32_t(r) < rank) sel_before += int(all[r][6]);
      }
      lse_t = UT.m + log2f(UT.z);
      lse_s = US.m + log2f(US.z);
      rkl0 = kLn2 * (US.b / US.z - (lse_s - lse_t));
    } else {
      lse_t = T_.m + log2f(T_.z);
      lse_s = S_.m + log2f(S_.z);
      rkl0 = kLn2 * (S_.b / S_.z - (lse_s - lse_t));
    }

    // ---- pass 2 (shared memory): loss terms and the gradient -----------------
    const float dl = lse_t - lse_s;
    const float wf = a.type == AQFQ_KD_KL ? 1.0f : a.type == AQFQ_KD_RKL ? 0.0f : 1.0f - conf;
    const float wr = a.type == AQFQ_KD_KL ? 0.0f : a.type == AQFQ_KD_RKL ? 1.0f : conf;
    float fs = 0.0f, rs = 0.0f;
    for (int v = tid; v < nvec; v += kThr) {
      const uint4 w = *reinterpret_cast<const uint4*>(tsl + 8 * v);
      const uint4 x = *reinterpret_cast<const uint4*>(ssl + 8 * v);
      const uint32_t tw[4] = {w.x, w.y, w.z, w.w}, sw[4] = {x.x, x.y, x.z, x.w};
      float g[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        g[j] = 0.0f;
        if (TOPK && !selected(8 * v + j, okey(j & 1 ? tw[j >> 1] >> 16 : tw[j >> 1]))) continue;
        const float t = bf16f(tw[j >> 1], j & 1), s = bf16f(sw[j >> 1], j & 1);
        const float pt = ex2(__fmaf_rn(t, ks, -lse_t)), ps = ex2(__fmaf_rn(s, ks, -lse_s));
        // log p_t - log p_s in nats
        const float dn = kLn2 * (__fmul_rn(__fsub_rn(t, s), ks) - dl);
        fs = __fadd_rn(fs, __fmaf_rn(pt, dn, ps - pt));
        rs = __fadd_rn(rs, __fmaf_rn(-ps, dn, pt - ps));
        if (drow)
          g[j] = mse ? gsc * __fsub_rn(s, t) : gsc * (wf * (ps - pt) + wr * ps * (-dn - rkl0));
      }
      if (drow)
        st_stream16(drow + 8 * v, make_uint4(pack2(g[1], g[0]), pack2(g[3], g[2]), pack2(g[5], g[4]),
                                             pack2(g[7], g[6])));
    }
    {
      float v2[2] = {fs, rs};
      block_sum<2>(v2, sh);
      const float mine[2] = {v2[0], v2[1]};
      float all[kCl][2];
      cluster_exchange<2>(mine, all, sh, par);
      float F = 0.0f, R = 0.0f;
#pragma unroll
      for (int r = 0; r < kCl; ++r) {
        F = __fadd_rn(F, all[r][0]);
        R = __fadd_rn(R, all[r][1]);
      }
      F = a.tau2 * F;
      R = a.tau2 * R;
      if (rank == 0 && tid == 0) {
        const float loss = a.type == AQFQ_KD_KL    ? F
                           : a.type == AQFQ_KD_RKL ? R
                           : a.type == AQFQ_KD_MSE ? SE / float(a.V)
                                                   : conf * R + (1.0f - conf) * F;
        a.tok[3 * row] = loss;
        a.tok[3 * row + 1] = F;
        a.tok[3 * row + 2] = R;
        if (a.token_loss) a.token_loss[row] = loss;
      }
    }
    if (TOPK && a.topk_idx) {  // the support in ascending vocabulary order
      int32_t* out = a.topk_idx + row * a.K + sel_before;
      const int32_t vb = int32_t(v0);
      const int room = a.K - sel_before;  // a support larger than K is never written past the row
      ordered_scan(
          tsl, nvec, selected,
          [&](int i, int pos) {
            if (pos < room) out[pos] = vb + i;
          },
          sh);
    }
  }
  // no CTA leaves while a peer may still read its shared memory
  cluster_sync();
}

// number of positions whose label lies in [0, V)
__global__ void kd_count_kernel(const int32_t* labels, int64_t T, int64_t V, int32_t* out) {
  __shared__ int part[32];
  int c = 0;
  for (int64_t i = threadIdx.x; i < T; i += blockDim.x) c += (labels[i] >= 0 && labels[i] < V);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, d);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int k = 0; k < int(blockDim.x >> 5); ++k) s += part[k];
    *out = s;
  }
}

// losses[k] = sum over positions of tok[:, k] / number of valid positions
// (ignored positions hold zeros); double accumulation, fixed order
__global__ void kd_mean_kernel(const float* tok, const int32_t* nvalid, int64_t T, float* losses) {
  __shared__ double part[32][3];
  double s[3] = {0.0, 0.0, 0.0};
  for (int64_t i = threadIdx.x; i < T; i += blockDim.x)
#pragma unroll
    for (int k = 0; k < 3; ++k) s[k] += double(tok[3 * i + k]);
#pragma unroll
  for (int k = 0; k < 3; ++k)
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) s[k] += __shfl_xor_sync(0xFFFFFFFFu, s[k], d);
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int k = 0; k < 3; ++k) part[threadIdx.x >> 5][k] = s[k];
  __syncthreads();
  if (threadIdx.x < 3) {
    double t = 0.0;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) t += part[w][threadIdx.x];
    const int n = T > 0 ? *nvalid : 0;
    losses[threadIdx.x] = n > 0 ? float(t / double(n)) : 0.0f;
  }
}

}  // namespace
}  // namespace aqfq

// ---- host side -------------------------------------------------------------

namespace {

using namespace aqfq;

constexpr size_t kWsHead = 256;  // workspace: int32 valid count, then tok [T, 3]

size_t kd_smem_bytes(int32_t S, bool topk) {
  return sizeof(KdShared) + (topk ? size_t(kHist1) * 4 : 0) + size_t(S) * 4;
}

int max_smem_optin() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  return v;
}

template <bool TOPK>
cudaError_t launch_kd(const KdArgs& a, size_t smem, cudaStream_t st) {
  auto kern = kd_loss_kernel<TOPK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
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

bool al(const void* p, uintptr_t b) { return (reinterpret_cast<uintptr_t>(p) & (b - 1)) == 0; }

}  // namespace

extern "C" size_t aqfq_kd_workspace_bytes(int64_t T) {
  if (T < 0) return 0;
  return kWsHead + ((size_t(T) * 12 + 255) / 256) * 256;
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
  if (smem > size_t(optin)) return AQFQ_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* nvalid = static_cast<int32_t*>(workspace);
  float* tok = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kWsHead);
  kd_count_kernel<<<1, 1024, 0, st>>>(labels, T, V, nvalid);
  if (cudaGetLastError() != cudaSuccess) return AQFQ_ERR_CUDA;
  if (T > 0) {
    KdArgs a;
    a.s = static_cast<const uint16_t*>(student);
    a.t = static_cast<const uint16_t*>(teacher);
    a.labels = labels;
    a.nvalid = nvalid;
    a.tok = tok;
    a.token_loss = token_loss;
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
    const cudaError_t e = use_topk ? launch_kd<true>(a, smem, st) : launch_kd<false>(a, smem, st);
    if (e != cudaSuccess) return AQFQ_ERR_CUDA;
  }
  kd_mean_kernel<<<1, 1024, 0, st>>>(tok, nvalid, T, losses);
  return cudaGetLastError() == cudaSuccess ? AQFQ_OK : AQFQ_ERR_CUDA;
}
