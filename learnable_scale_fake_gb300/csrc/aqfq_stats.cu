// aqfq_stats.cu -- per-head min/max observer, per-head scale, scale init.
//
// Observer (msModelSlim guide, "FA3Quant" steps 3-4): x [T, H, D] BF16.  The
// threads used form a multiple of the chunks per token, so each thread always
// reads the same (head, column-chunk) position of successive tokens and keeps
// a running min/max in registers as order-preserving 16-bit keys (two packed
// per register, SIMD min/max).  Runs of lanes that share a head are merged by
// a segmented shuffle; one lane per run applies atomicMin/atomicMax to 32-bit
// order-preserving keys stored in the caller's min/max arrays.  min/max are
// order-independent, so the result is exact and reproducible.  Three
// stream-ordered launches: keys in (identity or the caller's running values),
// reduce, keys back to floats.
//
// Scale init ("QAT + DeepSpeed ZeRO-3", "Quantizer initial values": scale =
// max|W| / 448 for FP8; the same rule with 127 / 7 / 6 for the other grids):
// per-block and per-group scales are reduced by shuffles and stored directly;
// the other units zero their outputs, atomicMax the float bits of |x|
// (non-negative floats order like their bit patterns), then divide in place.
#include "aqfq_internal.h"

namespace aqfq {

namespace {

// order-preserving keys: -0 orders below +0, negatives below positives
__device__ __forceinline__ uint32_t key32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unkey32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// two BF16 patterns per register -> two 16-bit keys
__device__ __forceinline__ uint32_t key16x2(uint32_t w) {
  const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xFFFFu;
  return w ^ (neg | 0x80008000u);
}
__device__ __forceinline__ uint32_t bf16_of_key16(uint32_t k) {
  return (k & 0x8000u) ? (k ^ 0x8000u) : (k ^ 0xFFFFu);
}

__global__ void observer_keys_in(float* mn, float* mx, int64_t H, int accumulate) {
  for (int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; h < H;
       h += (int64_t)gridDim.x * blockDim.x) {
    const float lo = accumulate ? mn[h] : __int_as_float(0x7F800000);   // +inf
    const float hi = accumulate ? mx[h] : __int_as_float((int)0xFF800000u);  // -inf
    reinterpret_cast<uint32_t*>(mn)[h] = key32(lo);
    reinterpret_cast<uint32_t*>(mx)[h] = key32(hi);
  }
}

__global__ void observer_keys_out(float* mn, float* mx, int64_t H) {
  for (int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; h < H;
       h += (int64_t)gridDim.x * blockDim.x) {
    mn[h] = unkey32(reinterpret_cast<uint32_t*>(mn)[h]);
    mx[h] = unkey32(reinterpret_cast<uint32_t*>(mx)[h]);
  }
}

constexpr int kObsU = 4;

template <int L>
__global__ void __launch_bounds__(kThreads)
    observer_reduce(const uint8_t* x, uint64_t nchunks, uint32_t cpt, FastDiv cph, uint64_t used,
                    uint32_t* kmn, uint32_t* kmx) {
  constexpr int NW = LayT<L>::NW;
  const uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
  const bool active = j < used;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  int64_t head = -1;
  if (active) {
    head = fdiv((uint32_t)(j % cpt), cph);
    for (uint64_t c0 = j; c0 < nchunks; c0 += used * kObsU) {
      uint32_t w[kObsU][NW];
#pragma unroll
      for (int u = 0; u < kObsU; ++u) {
        const uint64_t c = c0 + u * used;
        if (c < nchunks) ld_chunk<L>(x, c, w[u]);
      }
#pragma unroll
      for (int u = 0; u < kObsU; ++u) {
        if (c0 + u * used < nchunks) {
#pragma unroll
          for (int i = 0; i < NW; ++i) {
            const uint32_t k = key16x2(w[u][i]);
            lo = __vminu2(lo, k);
            hi = __vmaxu2(hi, k);
          }
        }
      }
    }
  }
  // per-thread 16-bit keys -> 32-bit float keys (identity stays identity)
  const uint32_t lo16 = min(lo & 0xFFFFu, lo >> 16), hi16 = max(hi & 0xFFFFu, hi >> 16);
  uint32_t klo = 0xFFFFFFFFu, khi = 0u;
  if (active && lo16 != 0xFFFFu) klo = key32(__uint_as_float(bf16_of_key16(lo16) << 16));
  if (active && hi16 != 0u) khi = key32(__uint_as_float(bf16_of_key16(hi16) << 16));
  if (active && lo16 == 0xFFFFu && hi16 == 0u) head = -1;  // saw no element
  // segmented merge of runs of lanes with the same head
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t oh = __shfl_down_sync(0xFFFFFFFFu, head, off);
    const uint32_t ol = __shfl_down_sync(0xFFFFFFFFu, klo, off);
    const uint32_t oh2 = __shfl_down_sync(0xFFFFFFFFu, khi, off);
    if (lane + off < 32 && oh == head) {
      klo = min(klo, ol);
      khi = max(khi, oh2);
    }
  }
  const int64_t prev = __shfl_up_sync(0xFFFFFFFFu, head, 1);
  if (head >= 0 && (lane == 0 || prev != head)) {
    atomicMin(kmn + head, klo);
    atomicMax(kmx + head, khi);
  }
}

__global__ void minmax_scale_kernel(const float* mn, const float* mx, int64_t H, float qmax,
                                    float* scale) {
  for (int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; h < H;
       h += (int64_t)gridDim.x * blockDim.x) {
    scale[h] = __fdiv_rn(fmaxf(fabsf(mn[h]), fabsf(mx[h])), qmax);
  }
}

// ---- scale init -----------------------------------------------------------

struct InitArgs {
  const uint8_t* x;
  uint32_t* sbits;  // scale array viewed as bits (NULL: NVFP4 dynamic)
  uint32_t* tbits;  // tensor-scale array viewed as bits (NVFP4 only)
  int64_t batch, rows;
  uint32_t cpb;
  FastDiv cpr;
  int lg;
  float qmax;
};

// Units of 1 << lg aligned lanes (NVFP4 blocks, groups): butterfly max, the
// first lane of the unit stores amax / qmax.  The NVFP4 tensor amax still goes
// through one atomicMax per warp.
template <bool NVFP4, int L>
__global__ void __launch_bounds__(kThreads) amax_direct_kernel(const InitArgs a) {
  constexpr int NW = LayT<L>::NW;
  const int lane = threadIdx.x & 31;
  const int width = 1 << a.lg;
  float* scale = reinterpret_cast<float*>(a.sbits);
  for (int64_t b = blockIdx.y; b < a.batch; b += gridDim.y) {
    const uint64_t base = (uint64_t)b * a.cpb;
    uint32_t tmax = 0;
    for (uint64_t c0 = (uint64_t)blockIdx.x * kThreads; c0 < a.cpb;
         c0 += (uint64_t)gridDim.x * kThreads) {
      const uint64_t c = c0 + threadIdx.x;
      uint32_t am = 0;
      if (c < a.cpb) {
        uint32_t w[NW];
        ld_chunk<L>(a.x, base + c, w);
        am = __float_as_uint(chunk_amax(w));
      }
      tmax = max(tmax, am);
      if (scale) {
        for (int off = 1; off < width; off <<= 1) am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
        if (c < a.cpb && (lane & (width - 1)) == 0)
          scale[(base + c) >> a.lg] = __fdiv_rn(__uint_as_float(am), a.qmax);
      }
    }
    if constexpr (NVFP4) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = max(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, off));
      if (lane == 0) atomicMax(a.tbits + b, tmax);
    }
  }
}

template <int GRAN, int L>
__global__ void __launch_bounds__(kThreads) amax_kernel(const InitArgs a) {
  constexpr int NW = LayT<L>::NW;
  const int lane = threadIdx.x & 31;
  for (int64_t b = blockIdx.y; b < a.batch; b += gridDim.y) {
    const uint64_t base = (uint64_t)b * a.cpb;
    uint32_t tmax = 0;
    for (uint64_t c0 = (uint64_t)blockIdx.x * kThreads; c0 < a.cpb;
         c0 += (uint64_t)gridDim.x * kThreads) {
      const uint64_t c = c0 + threadIdx.x;
      uint32_t am = 0;
      int64_t unit = -1;
      if (c < a.cpb) {
        uint32_t w[NW];
        ld_chunk<L>(a.x, base + c, w);
        am = __float_as_uint(chunk_amax(w));
        if constexpr (GRAN == G_TENSOR) unit = b;
        else if constexpr (GRAN == G_ROW) unit = b * a.rows + fdiv((uint32_t)c, a.cpr);
        else if constexpr (GRAN == G_HEAD) unit = fdiv((uint32_t)c, a.cpr);
        else unit = (int64_t)((base + c) >> a.lg);
      }
      tmax = max(tmax, am);
      if (a.sbits) {
        // segmented max over runs of lanes with the same unit
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int64_t ou = __shfl_down_sync(0xFFFFFFFFu, unit, off);
          const uint32_t oa = __shfl_down_sync(0xFFFFFFFFu, am, off);
          if (lane + off < 32 && ou == unit) am = max(am, oa);
        }
        const int64_t prev = __shfl_up_sync(0xFFFFFFFFu, unit, 1);
        if (unit >= 0 && (lane == 0 || prev != unit)) atomicMax(a.sbits + unit, am);
      }
    }
  }
}

__global__ void divide_in_place(float* v, int64_t n, float d) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    v[i] = __fdiv_rn(v[i], d);
}

unsigned small_grid(int64_t n) {
  int64_t b = (n + 255) / 256;
  if (b < 1) b = 1;
  if (b > 4096) b = 4096;
  return (unsigned)b;
}

// scale-init kernels of 16-element-chunk layouts
template <int L>
void init_launch(const Problem& p, const InitArgs& a, dim3 grid, bool nvfp4, bool direct,
                 cudaStream_t st) {
  if (nvfp4) {
    amax_direct_kernel<true, L><<<grid, kThreads, 0, st>>>(a);
  } else if (direct) {
    amax_direct_kernel<false, L><<<grid, kThreads, 0, st>>>(a);
  } else {
    switch (p.gran) {
      case G_TENSOR: amax_kernel<G_TENSOR, L><<<grid, kThreads, 0, st>>>(a); break;
      case G_ROW: amax_kernel<G_ROW, L><<<grid, kThreads, 0, st>>>(a); break;
      case G_HEAD: amax_kernel<G_HEAD, L><<<grid, kThreads, 0, st>>>(a); break;
      default: amax_kernel<G_GROUP, L><<<grid, kThreads, 0, st>>>(a); break;
    }
  }
}

template <int L>
void observer_launch(const uint8_t* x, uint64_t nchunks, uint32_t cpt, FastDiv cph, uint32_t* kmn,
                     uint32_t* kmx, cudaStream_t st) {
  // threads used: one wave of the kernel's resident CTAs, as a multiple of
  // the chunks per token
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, observer_reduce<L>, kThreads, 0) !=
          cudaSuccess || occ < 1)
    occ = 1;
  uint64_t want = uint64_t(sm_count()) * occ * kThreads;
  if (want > nchunks) want = nchunks;
  uint64_t used = want / cpt * cpt;
  if (used < cpt) used = cpt;
  const uint64_t blocks = (used + kThreads - 1) / kThreads;
  observer_reduce<L><<<(unsigned)blocks, kThreads, 0, st>>>(x, nchunks, cpt, cph, used, kmn, kmx);
}

}  // namespace

cudaError_t launch_observer(const void* x, int64_t T, int64_t H, int64_t D, int lay, float* mn,
                            float* mx, int accumulate, cudaStream_t st) {
  if (H == 0) return cudaSuccess;
  observer_keys_in<<<small_grid(H), 256, 0, st>>>(mn, mx, H, accumulate);
  const uint32_t ce = lay == L_8 ? 8 : 16;
  const uint64_t cpt = uint64_t(H) * uint64_t(D / ce);
  const uint64_t nchunks = uint64_t(T) * cpt;
  if (nchunks > 0) {
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const FastDiv cph = make_fastdiv((uint32_t)(D / ce));
    uint32_t* kmn = reinterpret_cast<uint32_t*>(mn);
    uint32_t* kmx = reinterpret_cast<uint32_t*>(mx);
    switch (lay) {
      case L_32: observer_launch<L_32>(xb, nchunks, (uint32_t)cpt, cph, kmn, kmx, st); break;
      case L_16: observer_launch<L_16>(xb, nchunks, (uint32_t)cpt, cph, kmn, kmx, st); break;
      default: observer_launch<L_8>(xb, nchunks, (uint32_t)cpt, cph, kmn, kmx, st); break;
    }
  }
  observer_keys_out<<<small_grid(H), 256, 0, st>>>(mn, mx, H);
  return cudaGetLastError();
}

cudaError_t launch_minmax_scale(const float* mn, const float* mx, int64_t H, float qmax,
                                float* scale, cudaStream_t st) {
  if (H == 0) return cudaSuccess;
  minmax_scale_kernel<<<small_grid(H), 256, 0, st>>>(mn, mx, H, qmax, scale);
  return cudaGetLastError();
}

cudaError_t launch_scale_init(const Problem& p, const void* x, float* scale, float* tscale,
                              cudaStream_t st) {
  const bool nvfp4 = p.fmt == F_NVFP4;
  const bool dyn = nvfp4 && p.mode == 1;
  // per-block / per-group scales are written directly, the others through atomics
  const bool direct = nvfp4 || p.gran == G_GROUP;
  int64_t nunit;
  if (nvfp4) nunit = dyn ? 0 : p.batch * int64_t(p.cpb);
  else if (p.gran == G_TENSOR) nunit = p.batch;
  else if (p.gran == G_ROW) nunit = p.batch * p.rows;
  else if (p.gran == G_HEAD) nunit = p.rows;
  else nunit = p.batch * p.rows * (p.K / p.group);
  cudaError_t e;
  if (!direct && nunit > 0 && (e = cudaMemsetAsync(scale, 0, size_t(nunit) * 4, st)) != cudaSuccess)
    return e;
  if (nvfp4 && p.batch > 0 && (e = cudaMemsetAsync(tscale, 0, size_t(p.batch) * 4, st)) != cudaSuccess)
    return e;
  if (p.batch > 0 && p.cpb > 0) {
    InitArgs a;
    a.x = static_cast<const uint8_t*>(x);
    a.sbits = dyn ? nullptr : reinterpret_cast<uint32_t*>(scale);
    a.tbits = reinterpret_cast<uint32_t*>(tscale);
    a.batch = p.batch;
    a.rows = p.rows;
    a.cpb = p.cpb;
    a.cpr = make_fastdiv(p.cpr);
    a.lg = 0;
    if (!nvfp4 && p.gran == G_GROUP) {
      while ((16 << a.lg) < p.group) ++a.lg;
    }
    a.qmax = nvfp4 ? 6.0f : (p.fmt == F_FP8 ? 448.0f : p.qmax);
    uint64_t gx = (uint64_t(p.cpb) + kThreads - 1) / kThreads;
    if (gx > 0x7FFFFFFFull) gx = 0x7FFFFFFFull;
    dim3 grid((unsigned)gx, (unsigned)(p.batch < 65535 ? p.batch : 65535), 1);
    if (p.lay == L_8) {
      switch (p.gran) {  // rows of 8 * odd elements: tensors, rows and heads only
        case G_TENSOR: amax_kernel<G_TENSOR, L_8><<<grid, kThreads, 0, st>>>(a); break;
        case G_ROW: amax_kernel<G_ROW, L_8><<<grid, kThreads, 0, st>>>(a); break;
        default: amax_kernel<G_HEAD, L_8><<<grid, kThreads, 0, st>>>(a); break;
      }
    } else if (p.lay == L_32) {
      init_launch<L_32>(p, a, grid, nvfp4, direct, st);
    } else {
      init_launch<L_16>(p, a, grid, nvfp4, direct, st);
    }
  }
  const float qmax = nvfp4 ? 6.0f : (p.fmt == F_FP8 ? 448.0f : p.qmax);
  if (!direct && nunit > 0) divide_in_place<<<small_grid(nunit), 256, 0, st>>>(scale, nunit, qmax);
  if (nvfp4 && p.batch > 0)
    divide_in_place<<<small_grid(p.batch), 256, 0, st>>>(tscale, p.batch, 448.0f * 6.0f);
  return cudaGetLastError();
}

}  // namespace aqfq
