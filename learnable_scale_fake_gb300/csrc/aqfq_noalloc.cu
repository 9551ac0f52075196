// aqfq_noalloc.cu -- aqfq_scale_grad_noalloc: the scale gradient for callers
// that cannot hand the library a scratch buffer.
//
// Some callers cannot allocate device memory at the point where they need the
// gradient: a plugin inside a host framework that owns all device memory
// through its own pool and exposes no allocation hook to the plugin, or a
// latency-critical path where a cudaMalloc (which may synchronise the device)
// is not acceptable.  The per-tensor and NVFP4 tensor-scale reductions of
// aqfq_scale_grad need device scratch for their per-CTA partial sums; this
// entry point takes it from a fixed array inside the library instead.
//
// The array below is 128 KiB (16384 doubles).  It lives in every GPU that
// loads the library until the process exits.  All calls share it: two calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it.  Each call overwrites every partial it later reads and
// zeroes the counter at its head on the stream, so nothing has to be cleared
// between calls.
//
// The first call on a device looks the array's device address up with
// cudaGetSymbolAddress while that device is current and caches it; make that
// first call before any stream capture.  No call allocates memory.
#include <mutex>

#include "aqfq.h"

namespace {

constexpr size_t kScratchBytes = size_t(128) << 10;
constexpr int kMaxDevices = 256;

__device__ __align__(256) double g_scale_grad_scratch[kScratchBytes / sizeof(double)];

std::mutex g_mu;
void* g_ptr[kMaxDevices];

// device address of the array on the current device (host code cannot use the
// symbol's name as an address); NULL on failure
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scale_grad_scratch) != cudaSuccess) return nullptr;
    g_ptr[dev] = p;
  }
  return g_ptr[dev];
}

}  // namespace

extern "C" aqfq_status aqfq_scale_grad_noalloc(const aqfq_qspec* spec, const void* x,
                                               const void* dy, int64_t batch, int64_t rows,
                                               int64_t K, const float* scale,
                                               const float* tensor_scale, float* dscale,
                                               float* dtensor_scale, void* dx, int accumulate,
                                               void* stream) {
  const size_t need = aqfq_scale_grad_workspace_bytes(spec, batch, rows, K);
  if (need > kScratchBytes) return AQFQ_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    ws = scratch_address();
    if (!ws) return AQFQ_ERR_CUDA;
  }
  return aqfq_scale_grad(spec, x, dy, batch, rows, K, scale, tensor_scale, dscale, dtensor_scale,
                         dx, accumulate, ws, need > 0 ? kScratchBytes : 0, stream);
}
