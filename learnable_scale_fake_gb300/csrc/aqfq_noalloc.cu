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
// loads the library until the process exits.  Three reductions take their
// scratch from it:
//   - per-tensor INT8 / INT4 / FP8 gradients and the NVFP4 tensor-scale
//     gradient: a 16-byte counter and one double per CTA and batch entry
//     (up to about 16380 batch entries);
//   - per-head gradients (x [T, H, D]): one double per thread used, and the
//     threads used are min(T * H * D / 16, one wave of the GPU), so a
//     per-head call fits only while T * H * D / 16 <= 16384 (262144 elements).
// Larger calls are rejected with AQFQ_ERR_WORKSPACE before anything runs.
// All calls share the array: two calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on it.  Each call
// overwrites every partial it later reads and zeroes the counter at its head
// on the stream, so nothing has to be cleared between calls.
//
// Host code cannot use the array's name as a device address: the address is
// looked up with cudaGetSymbolAddress while the device is current, once per
// device and context, and cached under the context's unique ID; after a
// device reset the new context has a new ID and the address is looked up
// again.  The first call on a device (or after a reset) may load the
// library's device code there, so make it before any stream capture.  No call
// allocates memory.
#include <cuda.h>

#include <mutex>

#include "aqfq.h"

namespace {

constexpr size_t kScratchBytes = size_t(128) << 10;
constexpr int kMaxDevices = 256;

__device__ __align__(256) double g_scale_grad_scratch[kScratchBytes / sizeof(double)];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

std::mutex g_mu;
void* g_ptr[kMaxDevices];
unsigned long long g_ctx[kMaxDevices];  // context ID the cached address belongs to

void* driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return p;
}

// unique ID of the context current on this thread; 0 when there is none or it
// cannot be read (the address is then looked up on every call)
unsigned long long current_context_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    get_current = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
    get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// device address of the array on the current device; NULL on failure
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long id = current_context_id();
  if (id != 0 && g_ptr[dev] && g_ctx[dev] == id) return g_ptr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scale_grad_scratch) != cudaSuccess || !p) return nullptr;
  g_ptr[dev] = p;
  g_ctx[dev] = current_context_id();  // the lookup made the device's context current
  return p;
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
