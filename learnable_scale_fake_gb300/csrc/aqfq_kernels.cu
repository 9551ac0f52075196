// aqfq_kernels.cu -- fake-quant forward and straight-through scale gradient.
//
// Forward (every format and granularity): one streaming kernel.  A CTA of 256
// threads covers 256*U consecutive chunks of one batch entry (one expert of a
// stack, gridDim.y over entries); each lane issues its U chunk loads (plus
// its scale) before computing, then writes one BF16 chunk and, on request,
// its packed codes.  No shared memory, no cross-lane traffic.
// Source of the operation: AngelSlim mcore_qad article, sections 1, 2.3, 2.4
// (whole-stack vectorised fake-quant) and 3 (formats).
//
// Gradient: the kernels of aqfq_grad.cuh, instantiated here without the
// forward output.
#include "aqfq_grad.cuh"

namespace aqfq {

namespace {

struct FwdArgs {
  const uint8_t* x;
  uint8_t* y;
  const float* scale;
  const float* tscale;
  uint8_t* codes;
  uint8_t* bcodes;
  int64_t batch, rows;
  uint32_t cpb;
  FastDiv cpr;
  int lg;
  IntRange ir;
};

template <int FMT, int GRAN, bool DYN, bool CODES, int U, int L>
__global__ void __launch_bounds__(kThreads) qdq_fwd_kernel(const FwdArgs a) {
  constexpr int NW = LayT<L>::NW;
  for (int64_t b = blockIdx.y; b < a.batch; b += gridDim.y) {
    const uint64_t base = (uint64_t)b * a.cpb;
    float g = 0.0f, st = 0.0f;
    if constexpr (FMT == F_NVFP4) g = __ldg(a.tscale + b);
    if constexpr (GRAN == G_TENSOR) st = __ldg(a.scale + b);
    for (uint64_t c0 = (uint64_t)blockIdx.x * (kThreads * U); c0 < a.cpb;
         c0 += (uint64_t)gridDim.x * (kThreads * U)) {
      uint32_t xw[U][NW];
      float sraw[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint64_t c = c0 + j * kThreads + threadIdx.x;
        sraw[j] = st;
        if (c < a.cpb) {
          const uint64_t gc = base + c;
          ld_chunk<L>(a.x, gc, xw[j]);
          if constexpr (FMT == F_NVFP4) {
            if constexpr (!DYN) sraw[j] = __ldg(a.scale + gc);
          } else if constexpr (GRAN == G_ROW) {
            sraw[j] = __ldg(a.scale + b * a.rows + fdiv((uint32_t)c, a.cpr));
          } else if constexpr (GRAN == G_HEAD) {
            sraw[j] = __ldg(a.scale + fdiv((uint32_t)c, a.cpr));
          } else if constexpr (GRAN == G_GROUP) {
            sraw[j] = __ldg(a.scale + (gc >> a.lg));
          }
        }
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint64_t c = c0 + j * kThreads + threadIdx.x;
        if (c >= a.cpb) continue;
        const uint64_t gc = base + c;
        float s = sraw[j];
        uint32_t ecode = 0;
        const float amax = chunk_amax(xw[j]);
        if constexpr (FMT == F_NVFP4) {
          const float sb = DYN ? __fdiv_rn(amax, 6.0f) : sraw[j];
          s = nvfp4_block_scale(sb, g, ecode);
        }
        uint32_t yw[NW], cw[4];
        const Divisor dv = make_divisor(s, amax);
        if (dv.fast) qdq_chunk_fast<FMT, CODES>(xw[j], dv, a.ir, yw, cw);
        else qdq_chunk<FMT, CODES>(xw[j], s, a.ir, yw, cw);
        if (a.y) st_chunk<L>(a.y, gc, yw);  // NULL: export of the codes only
        if constexpr (CODES) {
          st_codes<L, FMT == F_INT8 || FMT == F_FP8>(a.codes, gc, cw);
          if constexpr (FMT == F_NVFP4) a.bcodes[gc] = (uint8_t)ecode;
        }
      }
    }
  }
}

template <int FMT, int GRAN, bool DYN, bool CODES, int L>
void fwd_launch(const FwdArgs& a, cudaStream_t st) {
  constexpr int U = kFwdU;
  if (U > 1 && grad_unroll(a.cpb, a.batch, U) == U) {
    qdq_fwd_kernel<FMT, GRAN, DYN, CODES, U, L>
        <<<stream_grid(a.cpb, a.batch, U, 0), kThreads, 0, st>>>(a);
  } else {
    qdq_fwd_kernel<FMT, GRAN, DYN, CODES, 1, L>
        <<<stream_grid(a.cpb, a.batch, 1, 0), kThreads, 0, st>>>(a);
  }
}

// L_8 (rows of 8 * odd elements) exists only for the granularities whose unit
// is a whole row, a whole tensor or a head; the host checks never send a
// block or group format there
template <int FMT, bool CODES, int L>
void fwd_gran(const Problem& p, const FwdArgs& a, cudaStream_t st) {
  if constexpr (FMT == F_NVFP4) {
    static_assert(L != L_8, "NVFP4 blocks are 16 elements");
    if (p.mode == 1) fwd_launch<FMT, G_GROUP, true, CODES, L>(a, st);
    else fwd_launch<FMT, G_GROUP, false, CODES, L>(a, st);
  } else {
    switch (p.gran) {
      case G_TENSOR: fwd_launch<FMT, G_TENSOR, false, CODES, L>(a, st); break;
      case G_ROW: fwd_launch<FMT, G_ROW, false, CODES, L>(a, st); break;
      case G_GROUP:
        if constexpr (L != L_8) fwd_launch<FMT, G_GROUP, false, CODES, L>(a, st);
        break;
      default: fwd_launch<FMT, G_HEAD, false, CODES, L>(a, st); break;
    }
  }
}

template <int FMT, int L>
void fwd_codes(const Problem& p, const FwdArgs& a, cudaStream_t st) {
  if (a.codes) fwd_gran<FMT, true, L>(p, a, st);
  else fwd_gran<FMT, false, L>(p, a, st);
}

template <int FMT>
void fwd_lay(const Problem& p, const FwdArgs& a, cudaStream_t st) {
  if constexpr (FMT == F_NVFP4) {
    if (p.lay == L_32) fwd_codes<FMT, L_32>(p, a, st);
    else fwd_codes<FMT, L_16>(p, a, st);
  } else {
    switch (p.lay) {
      case L_32: fwd_codes<FMT, L_32>(p, a, st); break;
      case L_16: fwd_codes<FMT, L_16>(p, a, st); break;
      default: fwd_codes<FMT, L_8>(p, a, st); break;
    }
  }
}

}  // namespace

cudaError_t launch_qdq_fwd(const Problem& p, const void* x, const float* scale,
                           const float* tscale, void* y, uint8_t* codes, uint8_t* bcodes,
                           cudaStream_t st) {
  if (p.batch == 0 || p.cpb == 0) return cudaSuccess;
  FwdArgs a;
  a.x = static_cast<const uint8_t*>(x);
  a.y = static_cast<uint8_t*>(y);
  a.scale = scale;
  a.tscale = tscale;
  a.codes = codes;
  a.bcodes = bcodes;
  a.batch = p.batch;
  a.rows = p.rows;
  a.cpb = p.cpb;
  a.cpr = make_fastdiv(p.cpr ? p.cpr : 1);
  a.lg = p.gran == G_GROUP ? log2_exact(p.group / 16) : 0;
  if (p.fmt == F_NVFP4) a.lg = 0;
  a.ir = IntRange{p.qmin, p.qmax};
  switch (p.fmt) {
    case F_INT8: fwd_lay<F_INT8>(p, a, st); break;
    case F_INT4: fwd_lay<F_INT4>(p, a, st); break;
    case F_FP8: fwd_lay<F_FP8>(p, a, st); break;
    default: fwd_lay<F_NVFP4>(p, a, st); break;
  }
  return cudaGetLastError();
}

// Upper bounds over every instantiation (resident CTAs per SM <= 8), for the
// current device: the launches size their grids from the kernel's occupancy.
size_t grad_workspace_bytes(const Problem& p) {
  if (p.fmt != F_NVFP4 && p.gran == G_HEAD)
    return size_t(head_threads(p, kMaxCtasPerSm)) * sizeof(double);
  if (!grad_needs_partials(p) || p.batch == 0) return 0;
  // a 16-byte header (the CTAs' ticket), then the partials
  return 16 + size_t(p.batch) * size_t(grad_parts(p, kMaxCtasPerSm)) * sizeof(double);
}

cudaError_t launch_scale_grad(const Problem& p, const void* x, const void* dy, const float* scale,
                              const float* tscale, float* dscale, float* dtscale, void* dx,
                              int accumulate, double* ws, cudaStream_t st) {
  return launch_grad<false>(p, x, dy, scale, tscale, dscale, dtscale, dx, nullptr, accumulate, ws,
                            st);
}

}  // namespace aqfq
