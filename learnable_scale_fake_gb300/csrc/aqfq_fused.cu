// aqfq_fused.cu -- fake-quant forward and scale gradient in one pass.
//
// When the caller has the upstream gradient at the time it needs the
// forward's output (the forward recomputed in the backward pass, as under
// activation checkpointing: the weight's fake-quant output is needed for the
// input gradient while the weight gradient dW, the fake-quant's upstream
// gradient, needs no x_hat), one pass over x and dy writes x_hat and reduces
// the scale gradient: x is read once instead of twice and one launch replaces
// two.  The kernels are those of aqfq_grad.cuh with FWD = true; every output
// is bit for bit what aqfq_qdq_fwd and aqfq_scale_grad write.
#include "aqfq_grad.cuh"

namespace aqfq {

cudaError_t launch_qdq_fwd_grad(const Problem& p, const void* x, const void* dy,
                                const float* scale, const float* tscale, void* y, float* dscale,
                                float* dtscale, void* dx, int accumulate, double* ws,
                                cudaStream_t st) {
  return launch_grad<true>(p, x, dy, scale, tscale, dscale, dtscale, dx, y, accumulate, ws, st);
}

}  // namespace aqfq
