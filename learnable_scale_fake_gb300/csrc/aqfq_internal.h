// aqfq_internal.h -- launcher interface between the C ABI (aqfq_api.cu) and the
// kernel translation units.  Host-only declarations; arguments are already
// validated by the caller.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "aqfq_device.cuh"

namespace aqfq {

// A validated problem: x is [batch, rows, K] BF16, K % 8 == 0.  Chunks are
// 16 elements when K % 16 == 0, else 8 (per-tensor, per-channel and per-head
// INT8 / INT4 / FP8 only); lay is the chunk layout the launch uses (Lay).
struct Problem {
  int fmt, gran, group, mode;
  float qmin, qmax;
  int64_t batch, rows, K;
  int ce;        // elements per chunk: 16 or 8
  int lay;       // L_32, L_16 or L_8
  uint32_t cpb;  // chunks per batch entry = rows * K / ce
  uint32_t cpr;  // chunks per row = K / ce
};

int sm_count();

// forward (kernels.cu)
cudaError_t launch_qdq_fwd(const Problem& p, const void* x, const float* scale,
                           const float* tscale, void* y, uint8_t* codes, uint8_t* bcodes,
                           cudaStream_t st);

// scale gradient (kernels.cu); ws may be NULL when grad_workspace_bytes(p) == 0
size_t grad_workspace_bytes(const Problem& p);
cudaError_t launch_scale_grad(const Problem& p, const void* x, const void* dy, const float* scale,
                              const float* tscale, float* dscale, float* dtscale, void* dx,
                              int accumulate, double* ws, cudaStream_t st);

// forward and scale gradient in one pass (fused.cu); same workspace
cudaError_t launch_qdq_fwd_grad(const Problem& p, const void* x, const void* dy,
                                const float* scale, const float* tscale, void* y, float* dscale,
                                float* dtscale, void* dx, int accumulate, double* ws,
                                cudaStream_t st);

// statistics (stats.cu)
cudaError_t launch_observer(const void* x, int64_t T, int64_t H, int64_t D, int lay, float* mn,
                            float* mx, int accumulate, cudaStream_t st);
cudaError_t launch_minmax_scale(const float* mn, const float* mx, int64_t H, float qmax,
                                float* scale, cudaStream_t st);
cudaError_t launch_scale_init(const Problem& p, const void* x, float* scale, float* tscale,
                              cudaStream_t st);

}  // namespace aqfq
