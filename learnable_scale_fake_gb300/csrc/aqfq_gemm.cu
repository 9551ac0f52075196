// aqfq_gemm.cu -- fused NVFP4 weight fake-quant + grouped GEMM on tcgen05.
//
// For every expert e and its rows m in [off[e], off[e+1]) of X:
//   Y[m, n] = sum_k X[m, k] * W_hat_e[n, k],   W_hat_e = QDQ_NVFP4(W[e]; S[e], g[e])
// (AngelSlim mcore_qad article, section 2.4: the whole expert stack is
// fake-quantized, then one grouped GEMM computes every expert; here the
// fake-quantized weight tile is made in shared memory and never written to HBM).
//
// One CTA computes up to MT = 4 output tiles of 128 x 128 of one expert that
// share a column tile, K in steps of 64; the fake-quantized weight tile of a
// step feeds all of them (the fake-quant work per FLOP falls by the number of
// row tiles):
//   warp 0      TMA producer: X tiles [128 rows, 64] -> shared (128-byte swizzle)
//   warp 1      allocates the 512 TMEM columns (4 FP32 accumulators of 128 x
//               128); one lane issues tcgen05.mma (kind::f16, M=128, N=128,
//               K=16; 4 K-slices x up to 4 row tiles per step) and commits
//   warps 2-9   weight producers: load W chunks + block scales, fake-quantize
//               them (the same chunk arithmetic as aqfq_qdq_fwd) and store the
//               BF16 tile into shared memory in the 128-byte swizzle layout;
//               then the epilogue (TMEM -> registers -> BF16 -> Y), two warps
//               per TMEM lane quarter
// A 2-stage ring of (4 X tiles, 1 W_hat tile) = 80 KiB per stage; full barriers
// count the TMA bytes plus one arrival per producer warp, empty barriers are
// armed by tcgen05.commit.
// Every wait is bounded; on a timeout the CTA drains what it issued, frees
// its tensor memory, raises the caller's error flag and returns.
#include <cuda.h>

#include <mutex>

#include "aqfq.h"
#include "aqfq_internal.h"
#include "aqfq_sm100.cuh"

namespace aqfq {
namespace {

using namespace sm100;

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 2, MT = 4;
constexpr int kGemmThreads = 320;  // 10 warps
constexpr int kProducerThreads = 256;
constexpr uint32_t kTileBytes = BM * BK * 2;             // 16 KiB, one operand tile
constexpr uint32_t kStageA = MT * kTileBytes;            // 64 KiB of X per stage
constexpr uint32_t kTmemCols = MT * BN;                  // 512 columns
constexpr size_t kGemmSmem = 1024 + STAGES * (kStageA + kTileBytes) + 256;

struct GemmArgs {
  const uint8_t* w;       // [E, N, K] BF16
  const float* scale;     // [E, N, K/16]
  const float* tscale;    // [E]
  const int32_t* off;     // [E + 1]
  uint8_t* y;             // [total_M, N] BF16
  int32_t* err;           // optional error flag
  int64_t E, N, K;
  int64_t total_m;
};

struct __align__(8) GemmShared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t accum;
  uint32_t tmem;
  int32_t abort;
  int32_t expert, mtile;
};

__device__ __forceinline__ void set_abort(GemmShared* sh) {
  atomicExch(&sh->abort, 1);
}
__device__ __forceinline__ bool aborted(GemmShared* sh) {
  return *reinterpret_cast<volatile int32_t*>(&sh->abort) != 0;
}

// expert and row group of grid row `slot` (groups of MT x 128 rows, experts
// in order); one warp, result in *e / *mt (e = -1: no work)
__device__ void find_tile(const int32_t* off, int64_t E, int64_t total_m, int slot, int* e_out,
                          int* mt_out) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  for (int64_t e0 = 0; e0 < E; e0 += 32) {
    const int64_t e = e0 + lane;
    int t = 0;
    if (e < E) {
      int64_t lo = off[e], hi = off[e + 1];
      if (lo < 0) lo = 0;
      if (hi > total_m) hi = total_m;
      t = hi > lo ? int((hi - lo + MT * BM - 1) / (MT * BM)) : 0;  // groups of MT row tiles
    }
    int incl = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += v;
    }
    const int excl = incl - t;
    const bool hit = (e < E) && slot >= base + excl && slot < base + incl;
    const unsigned mask = __ballot_sync(0xFFFFFFFFu, hit);
    if (mask) {
      const int src = __ffs(mask) - 1;
      *e_out = (int)__shfl_sync(0xFFFFFFFFu, (int)e, src);
      *mt_out = slot - base - __shfl_sync(0xFFFFFFFFu, excl, src);
      return;
    }
    base += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  *e_out = -1;
  *mt_out = 0;
}

// one 16-element weight chunk: fake-quantize and store its 32 bytes into the
// swizzled tile (row n, 16-byte chunks 2j and 2j+1 of the row's 128 bytes)
__device__ __forceinline__ void qdq_store_chunk(const uint32_t (&xw)[8], float sb, float g,
                                                uint8_t* tile, int n, int j) {
  uint32_t ecode;
  const float s = nvfp4_block_scale(sb, g, ecode);
  uint32_t yw[8], cw[4];
  const Divisor dv = make_divisor(s, chunk_amax(xw));
  const IntRange r{-6.0f, 6.0f};
  if (dv.fast) qdq_chunk_fast<F_NVFP4, false>(xw, dv, r, yw, cw);
  else qdq_chunk<F_NVFP4, false>(xw, s, r, yw, cw);
  const int sw = n & 7;
  uint8_t* row = tile + n * 128;
  *reinterpret_cast<uint4*>(row + (((2 * j) ^ sw) * 16)) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
  *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ sw) * 16)) = make_uint4(yw[4], yw[5], yw[6], yw[7]);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_qdq_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* tiles_a = smem;                          // [STAGES][MT][16 KiB]
  uint8_t* tiles_b = smem + STAGES * kStageA;        // [STAGES][16 KiB]
  GemmShared* sh = reinterpret_cast<GemmShared*>(smem + STAGES * (kStageA + kTileBytes));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) {
    int e, mt;
    find_tile(a.off, a.E, a.total_m, blockIdx.y, &e, &mt);
    if (lane == 0) {
      sh->expert = e;
      sh->mtile = mt;
      sh->abort = 0;
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(&sh->full[s], 1 + kProducerThreads / 32);
        mbar_init(&sh->empty[s], 1);
      }
      mbar_init(&sh->accum, 1);
      fence_barrier_init();
      prefetch_tmap(&tmap_x);
    }
  }
  __syncthreads();
  const int e = sh->expert;
  if (e < 0) return;  // grid rows beyond the last tile: no work, nothing allocated
  const int mt = sh->mtile;
  if (warp == 1) tmem_alloc(&sh->tmem, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh->tmem;

  // rows [row0, row0 + rows_valid) of this expert, MT tiles at most
  const int64_t row0 = int64_t(a.off[e]) + int64_t(mt) * MT * BM;
  int64_t rows_valid = int64_t(a.off[e + 1]) - row0;
  if (rows_valid > MT * BM) rows_valid = MT * BM;
  if (row0 + rows_valid > a.total_m) rows_valid = a.total_m - row0;
  const int ntiles = int((rows_valid + BM - 1) / BM);  // 1..MT
  const int nt = blockIdx.x;
  const int KT = int(a.K / BK);

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      int issued = 0;
      for (int kt = 0; kt < KT && !aborted(sh); ++kt) {
        const int s = kt % STAGES;
        if (kt >= STAGES && !mbar_wait(&sh->empty[s], ((kt / STAGES) & 1) ^ 1)) {
          set_abort(sh);
          break;
        }
        mbar_arrive_expect_tx(&sh->full[s], kTileBytes * ntiles);
        for (int i = 0; i < ntiles; ++i)
          tma_load_2d(tiles_a + s * kStageA + i * kTileBytes, &tmap_x, &sh->full[s], kt * BK,
                      int32_t(row0 + i * BM));
        ++issued;
      }
      if (aborted(sh)) {
        // let the copies already issued land before the CTA's memory goes away
        for (int kt = (issued > STAGES ? issued - STAGES : 0); kt < issued; ++kt)
          mbar_wait(&sh->full[kt % STAGES], (kt / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % STAGES;
        if (aborted(sh) || !mbar_wait(&sh->full[s], (kt / STAGES) & 1)) {
          set_abort(sh);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sa = smem_u32(tiles_a + s * kStageA);
        const uint32_t sb = smem_u32(tiles_b + s * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t db = smem_desc_sw128(sb + kk * 32);
          for (int i = 0; i < ntiles; ++i)
            tc_mma_f16(tmem + uint32_t(i * BN), smem_desc_sw128(sa + i * kTileBytes + kk * 32), db,
                       idesc, (kt | kk) != 0);
        }
        tc_commit(&sh->empty[s]);
      }
      tc_commit(&sh->accum);
      if (!ok) mbar_wait(&sh->accum, 0);  // drain the MMAs already issued
    }
  } else {
    // ---- weight producers (fake-quant into shared memory) ----
    const int pt = threadIdx.x - 64;  // 0..255
    const float g = __ldg(a.tscale + e);
    const int64_t kb = a.K / 16;
    const uint8_t* wrow = a.w + (size_t(e) * a.N + size_t(nt) * BN) * size_t(a.K) * 2;
    const float* srow = a.scale + (size_t(e) * a.N + size_t(nt) * BN) * size_t(kb);
    int n_[2], j_[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = pt + i * kProducerThreads;
      n_[i] = c >> 2;
      j_[i] = c & 3;
    }
    uint32_t xw[2][8];
    float sbv[2];
    // prefetch step 0
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ld_stream(wrow + (size_t(n_[i]) * a.K + j_[i] * 16) * 2, xw[i]);
      sbv[i] = __ldg(srow + size_t(n_[i]) * kb + j_[i]);
    }
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % STAGES;
      uint32_t nx[2][8];
      float nsb[2];
      const bool more = kt + 1 < KT;
      if (more) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          ld_stream(wrow + (size_t(n_[i]) * a.K + size_t(kt + 1) * BK + j_[i] * 16) * 2, nx[i]);
          nsb[i] = __ldg(srow + size_t(n_[i]) * kb + size_t(kt + 1) * (BK / 16) + j_[i]);
        }
      }
      // lane 0 waits for the stage, the warp follows its verdict (warp-uniform)
      bool ok = true;
      if (lane == 0) {
        ok = !aborted(sh);
        if (ok && kt >= STAGES) ok = mbar_wait(&sh->empty[s], ((kt / STAGES) & 1) ^ 1);
        if (!ok) set_abort(sh);
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      __syncwarp();
      if (!ok) break;
      uint8_t* tile = tiles_b + s * kTileBytes;
#pragma unroll
      for (int i = 0; i < 2; ++i) qdq_store_chunk(xw[i], sbv[i], g, tile, n_[i], j_[i]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->full[s]);
      if (more) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
          for (int q = 0; q < 8; ++q) xw[i][q] = nx[i][q];
          sbv[i] = nsb[i];
        }
      }
    }
    // ---- epilogue: TMEM lane quarter = warp % 4, two warps per quarter ----
    {
      bool ok = true;
      if (lane == 0) {
        ok = !aborted(sh) && mbar_wait(&sh->accum, 0);
        if (!ok) set_abort(sh);
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      __syncwarp();
      if (ok) {
        tc_fence_after_sync();
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;  // 0 for warps 2-5, 1 for warps 6-9
#pragma unroll 1
        for (int p = half; p < ntiles * (BN / 32); p += 2) {
          const int i = p / (BN / 32), cc = p % (BN / 32);
          const int r = i * BM + q * 32 + lane;  // row within the group
          uint8_t* yrow = a.y + (size_t(row0 + r) * size_t(a.N) + size_t(nt) * BN) * 2;
          uint32_t v[32];
          tc_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + uint32_t(i * BN + cc * 32), v);
          tc_wait_ld();
          if (r < rows_valid) {
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[i] = pack_bf16x2(__uint_as_float(v[2 * i + 1]), __uint_as_float(v[2 * i]));
            uint4* dst = reinterpret_cast<uint4*>(yrow + cc * 64);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && aborted(sh) && a.err) atomicExch(a.err, 1);
}

// Diagnostic: one thread waits, through the same bounded wait as the GEMM's
// pipeline, for a barrier phase that nothing completes; when the wait gives
// up it raises *flag (the GEMM's timeout path sets its error flag the same way).
__global__ void wait_timeout_kernel(int32_t* flag, uint32_t polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait(&bar, 0, polls)) atomicExch(flag, 1);
}

// ---- host side -------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace
}  // namespace aqfq

extern "C" aqfq_status aqfq_grouped_qdq_gemm(const void* x, const int32_t* m_offsets,
                                             int64_t total_m, const void* w, const float* scale,
                                             const float* tensor_scale, int64_t E, int64_t N,
                                             int64_t K, void* y, int32_t* error_flag,
                                             void* stream) {
  using namespace aqfq;
  if (E < 1 || N < 0 || K < 0 || total_m < 0) return AQFQ_ERR_SHAPE;
  if (N % BN != 0 || K % BK != 0) return AQFQ_ERR_SHAPE;
  if (total_m > 0x7FFFFFFF || K > (int64_t(1) << 24) || N > (int64_t(1) << 24)) return AQFQ_ERR_SHAPE;
  const int64_t slots = (total_m + MT * BM - 1) / (MT * BM) + E;  // row groups, upper bound
  if (slots > 65535 || N / BN > 65535) return AQFQ_ERR_SHAPE;
  if (!m_offsets || !tensor_scale) return AQFQ_ERR_NULL;
  if (total_m == 0 || N == 0) return AQFQ_OK;
  if (K == 0) return AQFQ_ERR_SHAPE;  // an empty contraction would leave Y unwritten
  if (!x || !w || !scale || !y) return AQFQ_ERR_NULL;
  auto al = [](const void* p, uintptr_t b) { return (reinterpret_cast<uintptr_t>(p) & (b - 1)) == 0; };
  if (!al(x, 32) || !al(w, 32) || !al(y, 32) || !al(scale, 4) || !al(tensor_scale, 4) ||
      !al(m_offsets, 4) || (error_flag && !al(error_flag, 4)))
    return AQFQ_ERR_ALIGN;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return AQFQ_ERR_CUDA;
  CUtensorMap tm;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(total_m)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {BK, BM};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return AQFQ_ERR_CUDA;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(grouped_qdq_gemm_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(kGemmSmem));
  });
  if (attr_err != cudaSuccess) return AQFQ_ERR_CUDA;
  GemmArgs a;
  a.w = static_cast<const uint8_t*>(w);
  a.scale = scale;
  a.tscale = tensor_scale;
  a.off = m_offsets;
  a.y = static_cast<uint8_t*>(y);
  a.err = error_flag;
  a.E = E;
  a.N = N;
  a.K = K;
  a.total_m = total_m;
  dim3 grid(unsigned(N / BN), unsigned(slots), 1);
  grouped_qdq_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, static_cast<cudaStream_t>(stream)>>>(tm,
                                                                                                a);
  return cudaGetLastError() == cudaSuccess ? AQFQ_OK : AQFQ_ERR_CUDA;
}

extern "C" aqfq_status aqfq_selftest_wait_timeout(int32_t* flag, uint32_t polls, void* stream) {
  using namespace aqfq;
  if (!flag) return AQFQ_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(flag) & 3) != 0) return AQFQ_ERR_ALIGN;
  if (polls == 0 || polls > kWaitPolls) return AQFQ_ERR_SHAPE;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(flag, polls);
  return cudaGetLastError() == cudaSuccess ? AQFQ_OK : AQFQ_ERR_CUDA;
}
