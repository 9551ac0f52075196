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
// row tiles).  Warp w runs on scheduler w % 4; the MMA issuer's scheduler
// carries only the TMA warp and one fake-quant warp (arithmetic-heavy warps
// beside it starve its issue slots and stall the tensor pipe):
//   warp 1      allocates the 512 TMEM columns (4 FP32 accumulators of 128 x
//               128); one lane issues tcgen05.mma (kind::f16, M=128, N=128,
//               K=16; up to 4 row tiles x 4 K-slices per step, tile by tile)
//               and commits; it waits on its stages through try_wait
//   warp 5      TMA producer: X tiles [128 rows, 64] -> shared (128-byte swizzle)
//   warps 0, 2-4, 6-12, 14-16, 18, 19 (16 warps, five on each scheduler but
//               the MMA's)
//               weight producers: each thread loads one 16-element W chunk
//               and its block scale per step, fake-quantizes it (the same
//               chunk arithmetic as aqfq_qdq_fwd) and stores the BF16 values
//               into shared memory in the 128-byte swizzle layout
//   warps 4-11  epilogue (TMEM -> registers -> BF16 -> Y), two warps per TMEM
//               lane quarter (warp 0 sets up the barriers first)
// Two rings: X (2 stages of 4 tiles, 64 KiB each; full barriers count the TMA
// bytes) and W_hat (4 stages of 16 KiB; one arrival per producer warp), so the
// producers can run up to three k-steps ahead of the MMAs; empty barriers are
// armed by tcgen05.commit.
// Every CTA loads its own X tiles (column tiles of one row group read the
// same X rows from L2).
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

constexpr int BM = 128, BN = 128, BK = 64, MT = 4;
constexpr int XS = 2;  // X ring stages (MT tiles of 16 KiB each)
constexpr int WS = 4;  // fake-quantized weight ring stages (16 KiB each)
constexpr int kGemmThreads = 640;  // 20 warps
constexpr int kMmaWarp = 1, kTmaWarp = 5;
constexpr int kProducerThreads = 512;
constexpr int kChunksPerProducer = BN * BK / 16 / kProducerThreads;  // 16-element chunks per thread and k-step
static_assert(kChunksPerProducer * kProducerThreads * 16 == BN * BK, "producers cover the tile");
constexpr uint32_t kTileBytes = BM * BK * 2;             // 16 KiB, one operand tile
constexpr uint32_t kStageA = MT * kTileBytes;            // 64 KiB of X per stage
constexpr uint32_t kTmemCols = MT * BN;                  // 512 columns
constexpr size_t kScaleTab = 128 * 8;  // {S_hat, 1/S_hat} per non-negative E4M3 code
constexpr size_t kRings = size_t(XS) * kStageA + size_t(WS) * kTileBytes;  // 192 KiB
constexpr size_t kGemmSmem = 1024 + kRings + 256 + kScaleTab;

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
  uint64_t full_x[XS], empty_x[XS];  // TMA bytes / MMA commit
  uint64_t full_w[WS], empty_w[WS];  // one arrival per producer warp / MMA commit
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
// in order); one warp, result in *e / *mt (e = -1: no work).  Experts are
// taken 128 at a time, lane l holding experts l, l + 32, l + 64, l + 96: the
// offsets of a batch are loaded together, one round trip per 128 experts.
__device__ void find_tile(const int32_t* off, int64_t E, int64_t total_m, int slot, int* e_out,
                          int* mt_out) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  for (int64_t e0 = 0; e0 < E; e0 += 128) {
    int64_t lo[4], hi[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t e = e0 + q * 32 + lane;
      lo[q] = e < E ? int64_t(off[e]) : 0;
      hi[q] = e < E ? int64_t(off[e + 1]) : 0;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t e = e0 + q * 32 + lane;
      int t = 0;
      if (e < E) {
        int64_t l = lo[q], h = hi[q];
        if (l < 0) l = 0;
        if (h > total_m) h = total_m;
        t = h > l ? int((h - l + MT * BM - 1) / (MT * BM)) : 0;  // groups of MT row tiles
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
  }
  *e_out = -1;
  *mt_out = 0;
}

// ---- weight fake-quant in the producers ------------------------------------
// The same values as aqfq_qdq_fwd's NVFP4 chunk arithmetic, arranged for
// issue throughput (the producers' instruction count paces the main loop):
// the block scales S_hat = RN(dec(e) g) of the 128 non-negative E4M3 codes and
// their reciprocals come from a table built once per CTA (a negative code takes
// the IEEE path), the block-scale quotient
// S_b / g uses Markstein's correction with RN(1/g), and the per-element
// division and dequantisation run as packed f32x2 operations (IEEE
// round-to-nearest per lane, so every result is the scalar path's).

struct ScaleEntry {
  float s, r;  // S_hat and RN(1 / S_hat); r is NaN where the chunk takes the IEEE path
};

// S_hat for non-negative E4M3 code c and the reciprocal make_divisor would
// form (its fast range [2^-64, 2^64]; outside it r = NaN, which fails the
// chunk's range test)
__device__ __forceinline__ ScaleEntry scale_entry(uint32_t c, float g) {
  ScaleEntry e;
  e.s = __fmul_rn(dec_e4m3x2(c).x, g);
  const bool fast = (e.s >= 0x1p-64f) && (e.s <= 0x1p64f);
  e.r = fast ? __frcp_rn(e.s) : __int_as_float(0x7FC00000);
  return e;
}

// RN(S_b / g): q0 = RN(S_b rg), e = RN(S_b - q0 g) (exact), RN(q0 + e rg) is
// the IEEE quotient whenever 2^-30 <= |q0| <= 2^100 and g lies in
// [2^-64, 2^64] (rg = RN(1/g) there, NaN otherwise; ng = -g); every other case
// divides.  g = 0 gives the zero quotient, as nvfp4_block_scale does.
__device__ __forceinline__ float block_quotient(float sb, float g, float rg, float ng) {
  const float q0 = __fmul_rn(sb, rg);
  const float a = fabsf(q0);
  if (a >= 0x1p-30f && a <= 0x1p100f) return __fmaf_rn(__fmaf_rn(q0, ng, sb), rg, q0);
  return g != 0.0f ? __fdiv_rn(sb, g) : 0.0f;
}

// one 16-element weight chunk: fake-quantize and store its 32 bytes into the
// swizzled tile (row n, 16-byte chunks 2j and 2j+1 of the row's 128 bytes)
__device__ __forceinline__ void qdq_store_chunk(const uint32_t (&xw)[8], float sb, float g,
                                                float rg, float ng, const ScaleEntry* tab,
                                                uint8_t* tile, int n, int j) {
  const uint32_t ecode = cvt_e4m3x2(0.0f, block_quotient(sb, g, rg, ng)) & 0xFFu;
  ScaleEntry se;
  if (ecode < 128u) {
    se = tab[ecode];
  } else {  // a negative block scale: never the short path
    se.s = __fmul_rn(dec_e4m3x2(ecode).x, g);
    se.r = __int_as_float(0x7FC00000);
  }
  uint32_t aw[8], m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    aw[i] = xw[i] & 0x7FFF7FFFu;
    m = __vmaxu2(m, aw[i]);
  }
  const float amax = __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
  uint32_t yw[8];
  if (__fmul_rn(amax, se.r) <= 0x1p100f) {  // make_divisor's fast test (NaN r fails)
    const f2 R = mk2(se.r, se.r), S = mk2(se.s, se.s), NS = mk2(-se.s, -se.s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // |x| of the pair, divided (Markstein, as mdiv), rounded to E2M1, times S_hat
      const f2 x = mk2(__uint_as_float(aw[i] << 16), __uint_as_float(aw[i] & 0xFFFF0000u));
      const f2 q0 = mul2(x, R);
      const f2 v = fma2(fma2(q0, NS, x), R, q0);
      const uint32_t h = e2m1_q2(hi2(v), lo2(v));
      const f2 y = mul2(mk2(h2f(uint16_t(h & 0xFFFFu)), h2f(uint16_t(h >> 16))), S);
      yw[i] = pack_bf16x2(hi2(y), lo2(y)) | (xw[i] & 0x80008000u);
    }
  } else {
    uint32_t cw[4];
    qdq_chunk<F_NVFP4, false>(xw, se.s, IntRange{-6.0f, 6.0f}, yw, cw);
  }
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
  uint8_t* tiles_a = smem;                     // [XS][MT][16 KiB]
  uint8_t* tiles_b = smem + XS * kStageA;      // [WS][16 KiB]
  GemmShared* sh = reinterpret_cast<GemmShared*>(smem + kRings);
  ScaleEntry* stab = reinterpret_cast<ScaleEntry*>(smem + kRings + 256);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) {
    int e, mt;
    find_tile(a.off, a.E, a.total_m, blockIdx.y, &e, &mt);
    if (lane == 0) {
      sh->expert = e;
      sh->mtile = mt;
      sh->abort = 0;
      for (int s = 0; s < XS; ++s) {
        mbar_init(&sh->full_x[s], 1);
        mbar_init(&sh->empty_x[s], 1);
      }
      for (int s = 0; s < WS; ++s) {
        mbar_init(&sh->full_w[s], kProducerThreads / 32);
        mbar_init(&sh->empty_w[s], 1);
      }
      mbar_init(&sh->accum, 1);
      fence_barrier_init();
      prefetch_tmap(&tmap_x);
    }
  }
  __syncthreads();
  const int e = sh->expert;
  // grid rows beyond the last tile: no work, nothing allocated
  if (e < 0) return;
  const int mt = sh->mtile;
  if (warp == kMmaWarp) tmem_alloc(&sh->tmem, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh->tmem;

  // the expert's rows [lo, hi), offsets clamped to [0, total_m] as find_tile
  // counts them; this group: rows [row0, row0 + rows_valid), MT tiles at most
  // (an even spread of the tiles over the groups measured 1.8 % slower)
  int64_t lo = a.off[e], hi = a.off[e + 1];
  if (lo < 0) lo = 0;
  if (hi > a.total_m) hi = a.total_m;
  const int64_t row0 = lo + int64_t(mt) * MT * BM;
  int64_t rows_valid = hi - row0;
  if (rows_valid > MT * BM) rows_valid = MT * BM;
  const int ntiles = int((rows_valid + BM - 1) / BM);  // 1..MT
  const int nt = blockIdx.x;
  const int KT = int(a.K / BK);

  // producers: every warp but the MMA and TMA warps (1, 5, both on scheduler 1)
  // and two idle ones (13, 17): 5 on each other scheduler and one beside the MMA
  const bool producer = warp != kMmaWarp && warp != kTmaWarp && warp != 13 && warp != 17;
  if (warp == kTmaWarp) {
    // ---- TMA producer ----
    if (lane == 0) {
      int issued = 0;
      for (int kt = 0; kt < KT && !aborted(sh); ++kt) {
        const int s = kt % XS;
        if (kt >= XS && !mbar_wait(&sh->empty_x[s], ((kt / XS) & 1) ^ 1)) {
          set_abort(sh);
          break;
        }
        mbar_arrive_expect_tx(&sh->full_x[s], kTileBytes * ntiles);
        for (int i = 0; i < ntiles; ++i)
          tma_load_2d(tiles_a + s * kStageA + i * kTileBytes, &tmap_x, &sh->full_x[s], kt * BK,
                      int32_t(row0 + i * BM));
        ++issued;
      }
      if (aborted(sh)) {
        // let the copies already issued land before the CTA's memory goes away
        for (int kt = (issued > XS ? issued - XS : 0); kt < issued; ++kt)
          mbar_wait(&sh->full_x[kt % XS], (kt / XS) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      // descriptors of stage 0; a stage, row tile or K-slice offset adds to
      // the start-address field (addresses stay below 256 KiB: no carry)
      const uint64_t da0 = smem_desc_sw128(smem_u32(tiles_a));
      const uint64_t db0 = smem_desc_sw128(smem_u32(tiles_b));
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % XS, sw = kt % WS;
        if (aborted(sh) || !mbar_wait_suspend(&sh->full_x[s], (kt / XS) & 1) ||
            !mbar_wait_suspend(&sh->full_w[sw], (kt / WS) & 1)) {
          set_abort(sh);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t da = da0 + ((s * kStageA) >> 4), db = db0 + ((sw * kTileBytes) >> 4);
        // unrolled to MT with a guard: a loop bounded by the run-time tile
        // count issues the MMAs markedly slower
        // tile by tile, each tile's four K-slices back to back (issuing two
        // or three accumulators in turn measured up to twice as slow)
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          if (i < ntiles) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_f16(tmem + uint32_t(i * BN), da + ((i * kTileBytes + kk * 32) >> 4),
                         db + ((kk * 32) >> 4), idesc, (kt | kk) != 0);
          }
        }
        tc_commit(&sh->empty_x[s]);
        tc_commit(&sh->empty_w[sw]);
      }
      tc_commit(&sh->accum);
      if (!ok) mbar_wait(&sh->accum, 0);  // drain the MMAs already issued
    }
  } else if (producer) {
    // ---- weight producers (fake-quant into shared memory) ----
    const int pw = warp - (warp > kMmaWarp) - (warp > kTmaWarp) - (warp > 13) - (warp > 17);  // 0..15
    const int pt = pw * 32 + lane;                                                           // 0..511
    const int64_t kb = a.K / 16;
    const uint8_t* wrow = a.w + (size_t(e) * a.N + size_t(nt) * BN) * size_t(a.K) * 2;
    const float* srow = a.scale + (size_t(e) * a.N + size_t(nt) * BN) * size_t(kb);
    int n_[kChunksPerProducer], j_[kChunksPerProducer];
#pragma unroll
    for (int i = 0; i < kChunksPerProducer; ++i) {
      const int c = pt + i * kProducerThreads;
      n_[i] = c >> 2;
      j_[i] = c & 3;
    }
    uint32_t xw[kChunksPerProducer][8];
    float sbv[kChunksPerProducer];
    // step 0's weights and block scales are in flight while the table is built
#pragma unroll
    for (int i = 0; i < kChunksPerProducer; ++i) {
      ld_stream(wrow + (size_t(n_[i]) * a.K + j_[i] * 16) * 2, xw[i]);
      sbv[i] = __ldg(srow + size_t(n_[i]) * kb + j_[i]);
    }
    const float g = __ldg(a.tscale + e);
    const bool gfast = (g >= 0x1p-64f) && (g <= 0x1p64f);
    const float rg = gfast ? __frcp_rn(g) : __int_as_float(0x7FC00000), ng = -g;
    if (pt < 128) stab[pt] = scale_entry(uint32_t(pt), g);
    // the eight producer warps only: named barrier 1
    asm volatile("bar.sync 1, %0;" ::"n"(kProducerThreads) : "memory");
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % WS;
      uint32_t nx[kChunksPerProducer][8];
      float nsb[kChunksPerProducer];
      const bool more = kt + 1 < KT;
      if (more) {
#pragma unroll
        for (int i = 0; i < kChunksPerProducer; ++i) {
          ld_stream(wrow + (size_t(n_[i]) * a.K + size_t(kt + 1) * BK + j_[i] * 16) * 2, nx[i]);
          nsb[i] = __ldg(srow + size_t(n_[i]) * kb + size_t(kt + 1) * (BK / 16) + j_[i]);
        }
      }
      // lane 0 waits for the stage, the warp follows its verdict (warp-uniform)
      bool ok = true;
      if (lane == 0) {
        ok = !aborted(sh);
        if (ok && kt >= WS) ok = mbar_wait(&sh->empty_w[s], ((kt / WS) & 1) ^ 1);
        if (!ok) set_abort(sh);
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      __syncwarp();
      if (!ok) break;
      uint8_t* tile = tiles_b + s * kTileBytes;
#pragma unroll
      for (int i = 0; i < kChunksPerProducer; ++i) qdq_store_chunk(xw[i], sbv[i], g, rg, ng, stab, tile, n_[i], j_[i]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->full_w[s]);
      if (more) {
#pragma unroll
        for (int i = 0; i < kChunksPerProducer; ++i) {
#pragma unroll
          for (int q = 0; q < 8; ++q) xw[i][q] = nx[i][q];
          sbv[i] = nsb[i];
        }
      }
    }
  }
  if (warp >= 4 && warp < 12) {
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
        const int half = (warp - 4) >> 2;  // 0 for warps 4-7, 1 for warps 8-11
        // staging for 32 rows x 128 columns of BF16 (8 KiB per warp) in the
        // X ring, idle once the accumulators are complete; 16-byte unit c of
        // row r sits at unit c ^ (r % 16), so both the row-wise writes and the
        // column-wise reads below are free of bank conflicts
        uint8_t* stage = tiles_a + (warp - 4) * (32 * BN * 2);
#pragma unroll 1
        for (int i = half; i < ntiles; i += 2) {
          const int rb = i * BM + q * 32;  // first row of this warp's block within the group
          if (rb >= rows_valid) break;
#pragma unroll 1
          for (int cc = 0; cc < BN / 32; ++cc) {
            uint32_t v[32];
            tc_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + uint32_t(i * BN + cc * 32), v);
            tc_wait_ld();
            uint8_t* srow = stage + lane * (BN * 2);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * u + 1]), __uint_as_float(v[8 * u]));
              o.y = pack_bf16x2(__uint_as_float(v[8 * u + 3]), __uint_as_float(v[8 * u + 2]));
              o.z = pack_bf16x2(__uint_as_float(v[8 * u + 5]), __uint_as_float(v[8 * u + 4]));
              o.w = pack_bf16x2(__uint_as_float(v[8 * u + 7]), __uint_as_float(v[8 * u + 6]));
              *reinterpret_cast<uint4*>(srow + (((cc * 4 + u) ^ (lane & 15)) * 16)) = o;
            }
          }
          __syncwarp();
          // two rows of 256 bytes per instruction
#pragma unroll 4
          for (int t = 0; t < 16; ++t) {
            const int rr = 2 * t + (lane >> 4), c = lane & 15;
            const uint4 o = *reinterpret_cast<const uint4*>(stage + rr * (BN * 2) + ((c ^ (rr & 15)) * 16));
            if (rb + rr < rows_valid)
              *reinterpret_cast<uint4*>(a.y + (size_t(row0 + rb + rr) * size_t(a.N) + size_t(nt) * BN) * 2 +
                                        c * 16) = o;
          }
          __syncwarp();
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
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
  const unsigned ntn = unsigned(N / BN);
  grouped_qdq_gemm_kernel<<<dim3(ntn, unsigned(slots), 1), kGemmThreads, kGemmSmem,
                            static_cast<cudaStream_t>(stream)>>>(tm, a);
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
