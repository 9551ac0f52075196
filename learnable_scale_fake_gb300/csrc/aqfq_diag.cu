// aqfq_diag.cu -- aqfq_selftest_grid_codes: the grid rounding step of the
// fake-quant kernels applied to binary32 values given directly.
//
// Every forward and gradient kernel turns the quotient v = x / s into a code
// with the functions below (aqfq_device.cuh): the integer grids by clamping
// and round-half-even, E4M3 and E2M1 by the hardware saturating conversions
// on |v| with the sign of v put back on the code.  Exposing that step on its
// own lets a test compare it with the oracle for every binary32 value, which
// the BF16-input entry points cannot reach one value at a time.
#include "aqfq.h"
#include "aqfq_internal.h"

namespace aqfq {
namespace {

// one code per value: INT8 / FP8 a byte, INT4 / NVFP4 (E2M1) a nibble in the
// low four bits of its byte
template <int FMT>
__global__ void __launch_bounds__(kThreads) grid_codes_kernel(const float* v, int64_t n,
                                                              IntRange r, uint8_t* codes) {
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kThreads) {
    const float x = v[i];
    uint32_t code;
    if constexpr (FMT == F_INT8 || FMT == F_INT4) {
      int_round(x, r, code);
      code &= FMT == F_INT8 ? 0xFFu : 0xFu;
    } else {
      // the fast path's form: round |v|, then the sign of v on the code
      uint32_t c;
      fp_q2c<FMT>(0.0f, fabsf(x), c);
      const uint32_t sign = __float_as_uint(x) >> 31;
      code = (c & (FMT == F_FP8 ? 0xFFu : 0xFu)) | (sign << (FMT == F_FP8 ? 7 : 3));
    }
    codes[i] = (uint8_t)code;
  }
}

}  // namespace
}  // namespace aqfq

extern "C" aqfq_status aqfq_selftest_grid_codes(const aqfq_qspec* spec, const float* v, int64_t n,
                                                uint8_t* codes, void* stream) {
  using namespace aqfq;
  if (!spec) return AQFQ_ERR_NULL;
  if (n < 0) return AQFQ_ERR_SHAPE;
  if (n > 0 && (!v || !codes)) return AQFQ_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(v) & 3) != 0) return AQFQ_ERR_ALIGN;
  IntRange r{float(spec->qmin), float(spec->qmax)};
  switch (spec->fmt) {
    case AQFQ_INT8:
      if (!(spec->qmin >= -128 && spec->qmin < 0 && spec->qmax > 0 && spec->qmax <= 127))
        return AQFQ_ERR_UNSUPPORTED;
      break;
    case AQFQ_INT4:
      if (!(spec->qmin >= -8 && spec->qmin < 0 && spec->qmax > 0 && spec->qmax <= 7))
        return AQFQ_ERR_UNSUPPORTED;
      break;
    case AQFQ_FP8_E4M3:
    case AQFQ_NVFP4:
      break;
    default:
      return AQFQ_ERR_UNSUPPORTED;
  }
  if (n == 0) return AQFQ_OK;
  int64_t blocks = (n + kThreads - 1) / kThreads;
  if (blocks > 65536) blocks = 65536;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (spec->fmt) {
    case AQFQ_INT8: grid_codes_kernel<F_INT8><<<(unsigned)blocks, kThreads, 0, st>>>(v, n, r, codes); break;
    case AQFQ_INT4: grid_codes_kernel<F_INT4><<<(unsigned)blocks, kThreads, 0, st>>>(v, n, r, codes); break;
    case AQFQ_FP8_E4M3: grid_codes_kernel<F_FP8><<<(unsigned)blocks, kThreads, 0, st>>>(v, n, r, codes); break;
    default: grid_codes_kernel<F_NVFP4><<<(unsigned)blocks, kThreads, 0, st>>>(v, n, r, codes); break;
  }
  return cudaGetLastError() == cudaSuccess ? AQFQ_OK : AQFQ_ERR_CUDA;
}
