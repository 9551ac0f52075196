// aqfq_grad.cuh -- straight-through scale gradient kernels and their launch
// logic, shared by the gradient entry point (aqfq_kernels.cu) and the fused
// forward + gradient entry point (aqfq_fused.cu), which instantiate them with
// FWD = false and FWD = true in separate translation units.
//
// The gradient walks the chunks exactly as the forward does, recomputes v and
// q, forms dy * (clamped ? q : q - v) per element and reduces it
//   - per block / group (units of 16..512 elements = 1..32 aligned lanes):
//     the chunk's fixed-order sum in the lane (chunk_sum), xor-butterfly
//     across the unit's lanes, one store per unit (no atomics, no
//     workspace);
//   - per channel with long rows: one warp per row, per-lane double
//     accumulation of chunk sums, double butterfly;
//   - per tensor / NVFP4 tensor scale: per-CTA double partials into the
//     caller's workspace; the last CTA to finish (a ticket zeroed on the
//     stream before the launch) adds them, warp per entry, in fixed order;
//   - per head: per-thread double partials, a second kernel adds each head's.
// Every order is fixed, so results are bit-reproducible run to run.  With
// FWD the same pass also writes the forward's x_hat (bit for bit what
// aqfq_qdq_fwd writes), so x is read once for both.
// Source of the operation: AngelSlim mcore_qad article, sections 1 and 2.3
// (only the scales learn; the gradient flows to the scale through the
// fake-quant).
#pragma once

#include "aqfq_internal.h"

namespace aqfq {
namespace {

// Chunks per lane per iteration (U) and minimum resident CTAs per SM asked of
// the register allocator (MINB), per kernel instantiation, from GB300 sweeps
// on the workloads: resident warps beat deeper per-lane unrolling once the
// register cap makes the loop spill (INT4 group gradient of the expert stack:
// U = 2 at 4 CTAs per SM 0.262 ms; U = 3 at 4, spilling, 0.270; U = 3 at 3,
// 0.269).  The heavier instantiations (STE input gradient, dynamic block
// scale, partial sums) take one chunk per lane and fit 64 registers, 4 CTAs
// per SM, unfused; fused (FWD) they also hold x_hat and keep the allocator's
// choice.  The fused forward + gradient otherwise runs best at U = 2, 3 CTAs
// per SM.
template <int FMT, bool DYN, bool DX, int RED, bool FWD = false>
struct GradTune {
  static constexpr bool heavy = DX || DYN || RED != 0;
  static constexpr int U = heavy ? 1 : 2;
  static constexpr int MINB = heavy ? (FWD ? 1 : 4) : (FWD ? 3 : (FMT == F_NVFP4 ? 5 : 4));
};
template <bool DX, bool FWD = false>
struct RowTune {
  static constexpr int U = 2;
  static constexpr int MINB = (DX || FWD) ? 1 : 4;
};
constexpr int kFwdU = 2;

constexpr int kMaxCtasPerSm = 2048 / kThreads;  // resident 256-thread CTAs per SM, at most

// resident CTAs per SM of a kernel at 256 threads (at least 1)
template <typename Kernel>
int occupancy(Kernel kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

// x_hat of a chunk by IEEE division per element (the forward's exact path)
template <int FMT, int NW>
__device__ __forceinline__ void qdq_chunk_y(const uint32_t (&xw)[NW], float s, const IntRange& r,
                                            uint32_t (&yw)[NW]) {
  uint32_t cw[4];
  qdq_chunk<FMT, false>(xw, s, r, yw, cw);
}

struct GradArgs {
  const uint8_t* x;
  const uint8_t* dy;
  uint8_t* dx;
  uint8_t* y;           // FWD: the forward's x_hat, written by the same pass
  const float* scale;
  const float* tscale;
  float* dscale;
  double* ws;           // CTA partials [batch, nparts]
  unsigned* ticket;     // RED = 1: CTAs done (zeroed by the launch before the kernel)
  float* red_out;       // RED = 1: the per-batch-entry sums (dscale or the tensor-scale grads)
  int64_t batch, rows;
  uint32_t cpb;
  FastDiv cpr;
  int lg;
  IntRange ir;
  int accumulate;
  int nparts;
};

__device__ __forceinline__ void store_grad(float* p, float g, int accumulate) {
  *p = accumulate ? __fadd_rn(*p, g) : g;
}

// RED = 0: one scale per aligned run of (1 << lg) lanes, written directly.
// RED = 1: one scale (or NVFP4 tensor scale) per batch entry, CTA partials.
template <int FMT, int GRAN, bool DYN, bool DX, int RED, int U, int L, bool FWD>
__global__ void __launch_bounds__(kThreads, (GradTune<FMT, DYN, DX, RED, FWD>::MINB))
    scale_grad_kernel(const GradArgs a) {
  constexpr int NW = LayT<L>::NW;
  const int lane = threadIdx.x & 31;
  for (int64_t b = blockIdx.y; b < a.batch; b += gridDim.y) {
    const uint64_t base = (uint64_t)b * a.cpb;
    float g = 0.0f, st = 0.0f;
    if constexpr (FMT == F_NVFP4) g = __ldg(a.tscale + b);
    if constexpr (GRAN == G_TENSOR) st = __ldg(a.scale + b);
    double acc = 0.0;
    for (uint64_t c0 = (uint64_t)blockIdx.x * (kThreads * U); c0 < a.cpb;
         c0 += (uint64_t)gridDim.x * (kThreads * U)) {
      uint32_t xw[U][NW], dw[U][NW];
      float sraw[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint64_t c = c0 + j * kThreads + threadIdx.x;
        sraw[j] = st;
        if (c < a.cpb) {
          const uint64_t gc = base + c;
          ld_chunk<L>(a.x, gc, xw[j]);
          ld_chunk<L>(a.dy, gc, dw[j]);
          if constexpr (GRAN == G_GROUP && !DYN) sraw[j] = __ldg(a.scale + (gc >> a.lg));
        }
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint64_t c = c0 + j * kThreads + threadIdx.x;
        const bool valid = c < a.cpb;
        const uint64_t gc = base + c;
        float cs = 0.0f;
        float dec = 1.0f;
        if (valid) {
          float s = sraw[j];
          if constexpr (FMT == F_NVFP4) {
            uint32_t ecode;
            const float sb = DYN ? __fdiv_rn(chunk_amax(xw[j]), 6.0f) : sraw[j];
            s = nvfp4_block_scale(sb, g, ecode);
            dec = dec_e4m3x2(ecode).x;
          }
          uint32_t dxw[NW], yw[NW];
          const Divisor dv = make_divisor(s);
          bool slow = !dv.fast;
          if (dv.fast) {
            cs = grad_chunk_fast<FMT, DX, FWD>(xw[j], dw[j], dv, a.ir, dxw, yw);
            slow = isnan(cs);  // a quotient overflowed: redo the chunk exactly
          }
          if (slow) {
            cs = grad_chunk<FMT, DX>(xw[j], dw[j], s, a.ir, dxw);
            if constexpr (FWD) qdq_chunk_y<FMT>(xw[j], s, a.ir, yw);
          }
          if constexpr (DX) st_chunk<L>(a.dx, gc, dxw);
          if constexpr (FWD) st_chunk<L>(a.y, gc, yw);
        }
        if constexpr (RED == 0) {
          const int width = 1 << a.lg;
          for (int off = 1; off < width; off <<= 1)
            cs = __fadd_rn(cs, __shfl_xor_sync(0xFFFFFFFFu, cs, off));
          if (valid && (lane & (width - 1)) == 0) store_grad(a.dscale + (gc >> a.lg), cs, a.accumulate);
        } else {
          // NVFP4 dynamic: d S_hat / d g = dec(e_b) with the block code held fixed
          acc += (double)cs * (double)dec;
        }
      }
    }
    if constexpr (RED == 1) {
      __shared__ double red[kThreads / 32];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
      if (lane == 0) red[threadIdx.x >> 5] = acc;
      __syncthreads();
      if (threadIdx.x == 0) {
        double t = 0.0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) t += red[w];
        a.ws[b * a.nparts + blockIdx.x] = t;
      }
      __syncthreads();
    }
  }
  if constexpr (RED == 1) {
    // the last CTA to finish adds every entry's partials in a fixed order:
    // warp per entry, lane l takes partials l, l + 32, ..., then a butterfly
    __shared__ int last;
    if (threadIdx.x == 0) {
      __threadfence();  // this CTA's partials before its ticket
      last = atomicAdd(a.ticket, 1u) == gridDim.x * gridDim.y - 1u;
    }
    __syncthreads();
    if (last) {
      __threadfence();
      const volatile double* ws = a.ws;
      for (int64_t b = threadIdx.x >> 5; b < a.batch; b += kThreads / 32) {
        double t = 0.0;
        for (int i = lane; i < a.nparts; i += 32) t += ws[b * a.nparts + i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
        if (lane == 0) store_grad(a.red_out + b, (float)t, a.accumulate);
      }
    }
  }
}

// per-channel gradient for rows whose K is not a power of two <= 512: one warp
// per row, lanes stride over the row's chunks
template <int FMT, bool DX, int U, int L, bool FWD>
__global__ void __launch_bounds__(kThreads, (RowTune<DX, FWD>::MINB))
    scale_grad_row_kernel(const GradArgs a) {
  constexpr int NW = LayT<L>::NW;
  const int lane = threadIdx.x & 31;
  const int64_t nrows = a.batch * a.rows;
  const uint32_t cpr = a.cpr.d;
  for (int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); row < nrows;
       row += (int64_t)gridDim.x * (kThreads / 32)) {
    const float s = __ldg(a.scale + row);
    const Divisor dv = make_divisor(s);
    const uint64_t base = (uint64_t)row * cpr;
    double acc = 0.0;
    for (uint32_t c0 = 0; c0 < cpr; c0 += 32 * U) {
      uint32_t xw[U][NW], dw[U][NW];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + j * 32 + lane;
        if (c < cpr) {
          ld_chunk<L>(a.x, base + c, xw[j]);
          ld_chunk<L>(a.dy, base + c, dw[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + j * 32 + lane;
        if (c < cpr) {
          uint32_t dxw[NW], yw[NW];
          float cs = dv.fast ? grad_chunk_fast<FMT, DX, FWD>(xw[j], dw[j], dv, a.ir, dxw, yw) : 0.0f;
          if (!dv.fast || isnan(cs)) {
            cs = grad_chunk<FMT, DX>(xw[j], dw[j], s, a.ir, dxw);
            if constexpr (FWD) qdq_chunk_y<FMT>(xw[j], s, a.ir, yw);
          }
          acc += (double)cs;
          if constexpr (DX) st_chunk<L>(a.dx, base + c, dxw);
          if constexpr (FWD) st_chunk<L>(a.y, base + c, yw);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (lane == 0) store_grad(a.dscale + row, (float)acc, a.accumulate);
  }
}

// ---------------------------------------------------------------------------
// per-head gradient: x [T, H, D], one scale per head shared by all tokens.
// The threads used are a multiple of the chunks per token (cpt), so thread j
// always reads column-chunk j % cpt (one head) of successive tokens and sums
// its chunk gradients in double; ws[j] holds that partial.  A second kernel
// adds each head's partials in a fixed order.
// ---------------------------------------------------------------------------
struct HeadArgs {
  const uint8_t* x;
  const uint8_t* dy;
  uint8_t* dx;
  uint8_t* y;        // FWD: the forward's x_hat
  const float* scale;
  double* ws;
  uint64_t nchunks;  // T * cpt
  uint32_t cpt;
  FastDiv cph;       // chunks per head
  uint64_t used;     // threads with work (multiple of cpt)
  IntRange ir;
};

template <int FMT, bool DX, int L, bool FWD>
__global__ void __launch_bounds__(kThreads) scale_grad_head_kernel(const HeadArgs a) {
  constexpr int NW = LayT<L>::NW;
  const uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
  if (j >= a.used) return;
  const float s = __ldg(a.scale + fdiv((uint32_t)(j % a.cpt), a.cph));
  const Divisor dv = make_divisor(s);
  double acc = 0.0;
  for (uint64_t c0 = j; c0 < a.nchunks; c0 += 2 * a.used) {
    uint32_t xw[2][NW], dw[2][NW];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint64_t c = c0 + u * a.used;
      if (c < a.nchunks) {
        ld_chunk<L>(a.x, c, xw[u]);
        ld_chunk<L>(a.dy, c, dw[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint64_t c = c0 + u * a.used;
      if (c >= a.nchunks) continue;
      uint32_t dxw[NW], yw[NW];
      float cs = dv.fast ? grad_chunk_fast<FMT, DX, FWD>(xw[u], dw[u], dv, a.ir, dxw, yw) : 0.0f;
      if (!dv.fast || isnan(cs)) {
        cs = grad_chunk<FMT, DX>(xw[u], dw[u], s, a.ir, dxw);
        if constexpr (FWD) qdq_chunk_y<FMT>(xw[u], s, a.ir, yw);
      }
      acc += (double)cs;
      if constexpr (DX) st_chunk<L>(a.dx, c, dxw);
      if constexpr (FWD) st_chunk<L>(a.y, c, yw);
    }
  }
  a.ws[j] = acc;
}

// dscale[h] = sum over r < used / cpt, c < cph of ws[r * cpt + h * cph + c]:
// one block per head, thread t adding the head's partials i = t, t + blockDim,
// ... (i = r cph + c, carried along without division), then the warps' sums
// in warp order: a fixed order
__global__ void __launch_bounds__(kThreads) reduce_heads_kernel(const double* ws, uint64_t rounds,
                                                                uint32_t cpt, uint32_t cph,
                                                                int64_t H, float* out,
                                                                int accumulate) {
  __shared__ double red[kThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint64_t n = rounds * cph;
  const uint32_t dr = blockDim.x / cph, dc = blockDim.x % cph;
  for (int64_t h = blockIdx.x; h < H; h += gridDim.x) {
    double t = 0.0;
    uint64_t r = threadIdx.x / cph;
    uint32_t c = threadIdx.x % cph;
    for (uint64_t i0 = threadIdx.x; i0 < n; i0 += 8 * uint64_t(blockDim.x)) {
      double v[8];  // eight loads in flight, then added in order
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[k] = i0 + uint64_t(k) * blockDim.x < n ? ws[r * cpt + uint64_t(h) * cph + c] : 0.0;
        r += dr;
        c += dc;
        if (c >= cph) {
          c -= cph;
          ++r;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) t += v[k];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
    if (lane == 0) red[w] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
      double sum = 0.0;
      for (int k = 0; k < int(blockDim.x >> 5); ++k) sum += red[k];
      store_grad(out + h, (float)sum, accumulate);
    }
    __syncthreads();
  }
}

// threads used by the per-head gradient: one wave of `ctas_per_sm` CTAs per
// SM, rounded down to a multiple of the chunks per token (at least one token's
// worth), and no more than the chunks there are
uint64_t head_threads(const Problem& p, int ctas_per_sm) {
  const uint64_t cpt = p.cpr * uint64_t(p.rows);
  const uint64_t nchunks = uint64_t(p.batch) * cpt;
  if (cpt == 0) return 0;
  uint64_t want = uint64_t(sm_count()) * ctas_per_sm * kThreads;
  uint64_t used = want / cpt * cpt;
  if (used < cpt) used = cpt;
  if (used > nchunks) used = nchunks;
  return used;
}

// ---------------------------------------------------------------------------
// host-side dispatch
// ---------------------------------------------------------------------------

int log2_exact(int64_t v) {
  int l = 0;
  while ((int64_t(1) << l) < v) ++l;
  return (int64_t(1) << l) == v ? l : -1;
}

dim3 stream_grid(uint32_t cpb, int64_t batch, int U, int cap) {
  uint64_t gx = (uint64_t(cpb) + uint64_t(kThreads) * U - 1) / (uint64_t(kThreads) * U);
  if (gx < 1) gx = 1;
  if (cap > 0 && gx > uint64_t(cap)) gx = cap;
  if (gx > 0x7FFFFFFFull) gx = 0x7FFFFFFFull;
  uint64_t gy = batch < 65535 ? uint64_t(batch) : 65535ull;
  if (gy < 1) gy = 1;
  return dim3((unsigned)gx, (unsigned)gy, 1);
}

// unroll actually used by a gradient launch (U of the traits, or 1 when the
// batch entry has fewer than U * 256 chunks)
// U chunks per lane only when every batch entry has U * 256 chunks and the
// whole launch still fills one wave of one CTA per SM; small tensors take
// one chunk per lane (more CTAs in flight for the same bytes)
int grad_unroll(uint32_t cpb, int64_t batch, int U) {
  const uint64_t total = uint64_t(cpb) * uint64_t(batch < 65535 ? batch : 65535);
  const bool fill = total >= uint64_t(U) * kThreads * uint64_t(sm_count());
  return (cpb >= uint32_t(U) * kThreads && fill) ? U : 1;
}

bool grad_needs_partials(const Problem& p) {
  return (p.fmt == F_NVFP4 && p.mode == 1) || (p.fmt != F_NVFP4 && p.gran == G_TENSOR);
}

// every partial-sum (RED = 1) instantiation is "heavy": U = 1
static_assert(GradTune<F_NVFP4, true, false, 1>::U == 1 && GradTune<F_FP8, false, false, 1>::U == 1,
              "partial-sum kernels are launched with one chunk per lane");
// CTAs per batch entry of a partial-sum launch: one wave over all entries
// (ctas_per_sm resident CTAs on every SM), at most one per 256 chunks
int grad_parts(const Problem& p, int ctas_per_sm) {
  const int64_t entries = p.batch < 65535 ? p.batch : 65535;
  int64_t parts = int64_t(sm_count()) * ctas_per_sm / (entries > 0 ? entries : 1);
  const int64_t need = (int64_t(p.cpb) + kThreads - 1) / kThreads;
  if (parts > need) parts = need;
  if (parts < 1) parts = 1;
  return (int)parts;
}

// block-path lanes per unit (log2), or -1 when the row kernel is needed
int grad_unit_lg(const Problem& p) {
  if (p.fmt == F_NVFP4) return 0;
  if (p.gran == G_GROUP) return log2_exact(p.group / 16);
  if (p.gran == G_ROW) {
    const int l = log2_exact(p.cpr);
    return (l >= 0 && l <= 5) ? l : -1;
  }
  return 0;
}

// returns the CTAs per batch entry of a partial-sum launch (0 otherwise)
template <int FMT, int GRAN, bool DYN, bool DX, int RED, int L, bool FWD>
int grad_launch(const Problem& p, GradArgs a, cudaStream_t st) {
  constexpr int U = GradTune<FMT, DYN, DX, RED, FWD>::U;
  if constexpr (RED == 1) {
    auto k = scale_grad_kernel<FMT, GRAN, DYN, DX, RED, 1, L, FWD>;
    a.nparts = grad_parts(p, occupancy(k));
    k<<<stream_grid(a.cpb, a.batch, 1, a.nparts), kThreads, 0, st>>>(a);
    return a.nparts;
  } else {
    if (U > 1 && grad_unroll(a.cpb, a.batch, U) == U) {
      scale_grad_kernel<FMT, GRAN, DYN, DX, RED, U, L, FWD>
          <<<stream_grid(a.cpb, a.batch, U, 0), kThreads, 0, st>>>(a);
    } else {
      scale_grad_kernel<FMT, GRAN, DYN, DX, RED, 1, L, FWD>
          <<<stream_grid(a.cpb, a.batch, 1, 0), kThreads, 0, st>>>(a);
    }
    return 0;
  }
}

template <int FMT, bool DX, int L, bool FWD>
int grad_dispatch(const Problem& p, GradArgs a, cudaStream_t st) {
  if constexpr (FMT == F_NVFP4) {
    static_assert(L != L_8, "NVFP4 blocks are 16 elements");
    if (p.mode == 1) return grad_launch<FMT, G_GROUP, true, DX, 1, L, FWD>(p, a, st);
    return grad_launch<FMT, G_GROUP, false, DX, 0, L, FWD>(p, a, st);
  } else {
    if (p.gran == G_TENSOR) {
      return grad_launch<FMT, G_TENSOR, false, DX, 1, L, FWD>(p, a, st);
    } else if (a.lg >= 0) {  // per-group, or per-channel rows of 1..32 chunks (power of two)
      return grad_launch<FMT, G_GROUP, false, DX, 0, L, FWD>(p, a, st);
    } else {
      const int64_t nrows = p.batch * p.rows;
      int64_t blocks = (nrows + kThreads / 32 - 1) / (kThreads / 32);
      if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
      if (blocks < 1) blocks = 1;
      scale_grad_row_kernel<FMT, DX, RowTune<DX, FWD>::U, L, FWD><<<(unsigned)blocks, kThreads, 0, st>>>(a);
      return 0;
    }
  }
}

template <int FMT, int L, bool FWD>
int grad_dx(const Problem& p, const GradArgs& a, cudaStream_t st) {
  if (a.dx) return grad_dispatch<FMT, true, L, FWD>(p, a, st);
  return grad_dispatch<FMT, false, L, FWD>(p, a, st);
}

template <int FMT, bool FWD>
int grad_fmt(const Problem& p, const GradArgs& a, cudaStream_t st) {
  if constexpr (FMT == F_NVFP4) {
    if (p.lay == L_32) return grad_dx<FMT, L_32, FWD>(p, a, st);
    return grad_dx<FMT, L_16, FWD>(p, a, st);
  } else {
    switch (p.lay) {
      case L_32: return grad_dx<FMT, L_32, FWD>(p, a, st);
      case L_16: return grad_dx<FMT, L_16, FWD>(p, a, st);
      default: return grad_dx<FMT, L_8, FWD>(p, a, st);
    }
  }
}

// returns the threads used (one wave of the kernel's resident CTAs)
template <int FMT, bool DX, int L, bool FWD>
uint64_t head_launch(const Problem& p, HeadArgs a, cudaStream_t st) {
  auto k = scale_grad_head_kernel<FMT, DX, L, FWD>;
  a.used = head_threads(p, occupancy(k));
  const uint64_t blocks = (a.used + kThreads - 1) / kThreads;
  k<<<(unsigned)blocks, kThreads, 0, st>>>(a);
  return a.used;
}

template <int FMT, int L, bool FWD>
uint64_t head_dx(const Problem& p, const HeadArgs& a, cudaStream_t st) {
  if (a.dx) return head_launch<FMT, true, L, FWD>(p, a, st);
  return head_launch<FMT, false, L, FWD>(p, a, st);
}

template <int FMT, bool FWD>
uint64_t head_fmt(const Problem& p, const HeadArgs& a, cudaStream_t st) {
  switch (p.lay) {
    case L_32: return head_dx<FMT, L_32, FWD>(p, a, st);
    case L_16: return head_dx<FMT, L_16, FWD>(p, a, st);
    default: return head_dx<FMT, L_8, FWD>(p, a, st);
  }
}

template <bool FWD>
cudaError_t launch_head_grad(const Problem& p, const void* x, const void* dy, const float* scale,
                             float* dscale, void* dx, void* y, int accumulate, double* ws,
                             cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  if (p.batch == 0 || p.cpr == 0) {  // no elements: every head's gradient is an empty sum
    if (!accumulate) return cudaMemsetAsync(dscale, 0, size_t(p.rows) * sizeof(float), st);
    return cudaSuccess;
  }
  HeadArgs a;
  a.x = static_cast<const uint8_t*>(x);
  a.dy = static_cast<const uint8_t*>(dy);
  a.dx = static_cast<uint8_t*>(dx);
  a.y = static_cast<uint8_t*>(y);
  a.scale = scale;
  a.ws = ws;
  a.cpt = p.cpr * uint32_t(p.rows);
  a.nchunks = uint64_t(p.batch) * a.cpt;
  a.cph = make_fastdiv(p.cpr);
  a.used = 0;
  a.ir = int_range(p.qmin, p.qmax);
  uint64_t used;
  switch (p.fmt) {
    case F_INT8: used = head_fmt<F_INT8, FWD>(p, a, st); break;
    case F_INT4: used = head_fmt<F_INT4, FWD>(p, a, st); break;
    default: used = head_fmt<F_FP8, FWD>(p, a, st); break;
  }
  int64_t blocks = p.rows;  // one per head
  if (blocks > 65535) blocks = 65535;
  reduce_heads_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(ws, used / a.cpt, a.cpt, p.cpr,
                                                             p.rows, dscale, accumulate);
  return cudaGetLastError();
}

// The scale gradient (FWD: and the forward's x_hat in the same pass).
template <bool FWD>
cudaError_t launch_grad(const Problem& p, const void* x, const void* dy, const float* scale,
                        const float* tscale, float* dscale, float* dtscale, void* dx, void* y,
                        int accumulate, double* ws, cudaStream_t st) {
  if (p.fmt != F_NVFP4 && p.gran == G_HEAD)
    return launch_head_grad<FWD>(p, x, dy, scale, dscale, dx, y, accumulate, ws, st);
  const bool partials = grad_needs_partials(p);
  float* out = (p.fmt == F_NVFP4 && p.mode == 1) ? dtscale : dscale;
  if (p.batch == 0) return cudaSuccess;
  if (p.cpb == 0) {
    // empty rows: every gradient is an empty sum
    if (!accumulate) {
      size_t n = partials ? size_t(p.batch)
                          : (p.gran == G_ROW ? size_t(p.batch * p.rows) : 0);
      if (n) {
        cudaError_t e = cudaMemsetAsync(out, 0, n * sizeof(float), st);
        if (e != cudaSuccess) return e;
      }
    }
    return cudaGetLastError();
  }
  GradArgs a;
  a.x = static_cast<const uint8_t*>(x);
  a.dy = static_cast<const uint8_t*>(dy);
  a.dx = static_cast<uint8_t*>(dx);
  a.y = static_cast<uint8_t*>(y);
  a.scale = scale;
  a.tscale = tscale;
  a.dscale = dscale;
  a.ws = partials ? ws + 2 : ws;  // after the 16-byte ticket header
  a.ticket = partials ? reinterpret_cast<unsigned*>(ws) : nullptr;
  a.red_out = out;
  a.batch = p.batch;
  a.rows = p.rows;
  a.cpb = p.cpb;
  a.cpr = make_fastdiv(p.cpr);
  a.lg = grad_unit_lg(p);
  a.ir = int_range(p.qmin, p.qmax);
  a.accumulate = accumulate;
  a.nparts = 0;
  if (partials) {  // the ticket starts at zero on the stream, before the kernel
    cudaError_t e = cudaMemsetAsync(a.ticket, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
  }
  switch (p.fmt) {
    case F_INT8: grad_fmt<F_INT8, FWD>(p, a, st); break;
    case F_INT4: grad_fmt<F_INT4, FWD>(p, a, st); break;
    case F_FP8: grad_fmt<F_FP8, FWD>(p, a, st); break;
    default: grad_fmt<F_NVFP4, FWD>(p, a, st); break;
  }
  return cudaGetLastError();
}

}  // namespace
}  // namespace aqfq
