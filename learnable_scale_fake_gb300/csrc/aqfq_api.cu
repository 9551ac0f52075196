// aqfq_api.cu -- the extern "C" entry points of libaqfq: argument checks on the
// host, then the launches (include/aqfq.h documents every call).
#include <initializer_list>

#include "aqfq.h"
#include "aqfq_internal.h"

namespace aqfq {

// SM count of the current device, cached per device ordinal; 0 when the
// device cannot be queried (the entry points that size grids or workspaces
// from it then return AQFQ_ERR_CUDA instead of guessing)
int sm_count() {
  static int cache[256];  // 0 = not yet queried
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace aqfq

namespace {

using aqfq::Problem;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool pow2_in(int64_t v, int64_t lo, int64_t hi) {
  return v >= lo && v <= hi && (v & (v - 1)) == 0;
}

// Checks the spec and sizes; fills p (its chunk layout assumes 32-byte aligned
// data until choose_layout sees the pointers).  Pointer checks are done by the
// callers.
aqfq_status make_problem(const aqfq_qspec* sp, int64_t batch, int64_t rows, int64_t K,
                         Problem& p) {
  if (!sp) return AQFQ_ERR_NULL;
  if (batch < 0 || rows < 0 || K < 0 || K % 8 != 0) return AQFQ_ERR_SHAPE;
  const int ce = (K % 16 == 0) ? 16 : 8;
  if (ce == 8) {
    // rows of 8 * odd elements: only units that are whole rows, tensors or heads
    const bool fmt_ok = sp->fmt == AQFQ_INT8 || sp->fmt == AQFQ_INT4 || sp->fmt == AQFQ_FP8_E4M3;
    const bool gran_ok = sp->gran == AQFQ_PER_TENSOR || sp->gran == AQFQ_PER_CHANNEL ||
                         sp->gran == AQFQ_PER_HEAD;
    if (!fmt_ok || !gran_ok) return AQFQ_ERR_SHAPE;
  }
  if (rows > 0 && K / ce > int64_t(0xFFFFFFFF) / rows) return AQFQ_ERR_SHAPE;
  const int64_t cpb = rows * (K / ce);
  if (cpb > int64_t(0xFFFFFFFF)) return AQFQ_ERR_SHAPE;
  if (batch > 0 && cpb > 0 && batch > (int64_t(1) << 62) / (cpb * 32)) return AQFQ_ERR_SHAPE;
  p.ce = ce;
  p.lay = ce == 16 ? aqfq::L_32 : aqfq::L_8;
  p.fmt = sp->fmt;
  p.gran = sp->gran;
  p.group = sp->group;
  p.mode = sp->mode;
  p.batch = batch;
  p.rows = rows;
  p.K = K;
  p.cpb = uint32_t(cpb);
  p.cpr = uint32_t(K / ce);
  p.qmin = float(sp->qmin);
  p.qmax = float(sp->qmax);
  switch (sp->fmt) {
    case AQFQ_NVFP4:
      if (sp->gran != AQFQ_PER_GROUP || sp->group != 16) return AQFQ_ERR_UNSUPPORTED;
      if (sp->mode != AQFQ_SCALE_LEARNED && sp->mode != AQFQ_SCALE_DYNAMIC_BLOCK)
        return AQFQ_ERR_UNSUPPORTED;
      p.qmin = -6.0f;
      p.qmax = 6.0f;
      return AQFQ_OK;
    case AQFQ_INT8:
      if (!(sp->qmin >= -128 && sp->qmin < 0 && sp->qmax > 0 && sp->qmax <= 127))
        return AQFQ_ERR_UNSUPPORTED;
      break;
    case AQFQ_INT4:
      if (!(sp->qmin >= -8 && sp->qmin < 0 && sp->qmax > 0 && sp->qmax <= 7))
        return AQFQ_ERR_UNSUPPORTED;
      break;
    case AQFQ_FP8_E4M3:
      p.qmin = -448.0f;
      p.qmax = 448.0f;
      break;
    default:
      return AQFQ_ERR_UNSUPPORTED;
  }
  if (sp->mode != AQFQ_SCALE_LEARNED) return AQFQ_ERR_UNSUPPORTED;
  switch (sp->gran) {
    case AQFQ_PER_TENSOR:
    case AQFQ_PER_CHANNEL:
    case AQFQ_PER_HEAD:
      return AQFQ_OK;
    case AQFQ_PER_GROUP:
      if (!pow2_in(sp->group, 16, 512)) return AQFQ_ERR_UNSUPPORTED;
      if (K % sp->group != 0) return AQFQ_ERR_SHAPE;
      return AQFQ_OK;
    default:
      return AQFQ_ERR_UNSUPPORTED;
  }
}

bool byte_codes(const Problem& p) { return p.fmt == AQFQ_INT8 || p.fmt == AQFQ_FP8_E4M3; }

int64_t elems(const Problem& p) { return p.batch * int64_t(p.cpb) * p.ce; }

// The chunk layout for these BF16 tensors (NULL ones ignored): 16-element
// chunks with 256-bit accesses when every tensor is 32-byte aligned, with
// 128-bit accesses when one is only 16-byte aligned; 8-element chunks (K % 16
// != 0) need 16 bytes.  AQFQ_ERR_ALIGN below 16 bytes.
aqfq_status choose_layout(Problem& p, std::initializer_list<const void*> tensors) {
  bool a32 = true;
  for (const void* t : tensors) {
    if (!t) continue;
    if (!aligned(t, 16)) return AQFQ_ERR_ALIGN;
    a32 = a32 && aligned(t, 32);
  }
  if (p.ce == 16) p.lay = a32 ? aqfq::L_32 : aqfq::L_16;
  else p.lay = aqfq::L_8;
  return AQFQ_OK;
}

// codes: one byte per element (INT8 / FP8) or one nibble (INT4 / NVFP4); a
// chunk's codes are stored in one access
bool codes_aligned(const Problem& p, const void* codes) {
  const int bytes = byte_codes(p) ? p.ce : p.ce / 2;
  return aligned(codes, uintptr_t(bytes));
}

// number of learned scales (0 in NVFP4 dynamic mode)
int64_t scale_count(const Problem& p) {
  if (p.fmt == AQFQ_NVFP4) return p.mode == AQFQ_SCALE_DYNAMIC_BLOCK ? 0 : elems(p) / 16;
  switch (p.gran) {
    case AQFQ_PER_TENSOR: return p.batch;
    case AQFQ_PER_CHANNEL: return p.batch * p.rows;
    case AQFQ_PER_HEAD: return p.rows;
    default: return p.batch * p.rows * (p.K / p.group);
  }
}

// Pointers are required only for non-empty buffers (an empty tensor may be NULL).
aqfq_status check_scales(const Problem& p, const float* scale, const float* tscale) {
  const bool nvfp4 = p.fmt == AQFQ_NVFP4;
  if (nvfp4 && !tscale && p.batch > 0) return AQFQ_ERR_NULL;
  if (!scale && scale_count(p) > 0) return AQFQ_ERR_NULL;
  if (scale && !aligned(scale, 4)) return AQFQ_ERR_ALIGN;
  if (tscale && !aligned(tscale, 4)) return AQFQ_ERR_ALIGN;
  return AQFQ_OK;
}

aqfq_status finish(cudaError_t e) { return e == cudaSuccess ? AQFQ_OK : AQFQ_ERR_CUDA; }

}  // namespace

extern "C" {

const char* aqfq_status_string(aqfq_status s) {
  switch (s) {
    case AQFQ_OK: return "ok";
    case AQFQ_ERR_NULL: return "a required pointer is NULL";
    case AQFQ_ERR_SHAPE: return "invalid or unsupported size";
    case AQFQ_ERR_ALIGN: return "pointer misaligned";
    case AQFQ_ERR_UNSUPPORTED: return "unsupported format / granularity / mode";
    case AQFQ_ERR_WORKSPACE: return "workspace too small";
    case AQFQ_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

int aqfq_version(void) { return 100; }

aqfq_status aqfq_qdq_fwd(const aqfq_qspec* spec, const void* x, int64_t batch, int64_t rows,
                         int64_t K, const float* scale, const float* tensor_scale, void* y,
                         uint8_t* codes, uint8_t* block_codes, void* stream) {
  Problem p;
  aqfq_status s = make_problem(spec, batch, rows, K, p);
  if (s != AQFQ_OK) return s;
  const bool any = elems(p) > 0;
  if (any && (!x || (!y && !codes))) return AQFQ_ERR_NULL;
  if ((s = check_scales(p, scale, tensor_scale)) != AQFQ_OK) return s;
  if ((s = choose_layout(p, {x, y})) != AQFQ_OK) return s;
  if (codes && !codes_aligned(p, codes)) return AQFQ_ERR_ALIGN;
  if (block_codes && p.fmt != AQFQ_NVFP4) return AQFQ_ERR_UNSUPPORTED;
  if (codes && p.fmt == AQFQ_NVFP4 && !block_codes) return AQFQ_ERR_NULL;
  if (block_codes && !codes) return AQFQ_ERR_NULL;
  return finish(aqfq::launch_qdq_fwd(p, x, scale, tensor_scale, y, codes, block_codes,
                                     static_cast<cudaStream_t>(stream)));
}

aqfq_status aqfq_grouped_qdq(const aqfq_qspec* spec, const void* w, int64_t E, int64_t N,
                             int64_t K, const float* scale, const float* tensor_scale, void* y,
                             uint8_t* codes, uint8_t* block_codes, void* stream) {
  return aqfq_qdq_fwd(spec, w, E, N, K, scale, tensor_scale, y, codes, block_codes, stream);
}

size_t aqfq_scale_grad_workspace_bytes(const aqfq_qspec* spec, int64_t batch, int64_t rows,
                                       int64_t K) {
  Problem p;
  if (make_problem(spec, batch, rows, K, p) != AQFQ_OK) return 0;
  if (aqfq::sm_count() <= 0) return 0;
  return aqfq::grad_workspace_bytes(p);
}

}  // extern "C"

namespace {

// The checks shared by the gradient and the fused forward + gradient: fills p
// and leaves the launch to the caller.  y (fused only) joins the layout choice.
aqfq_status check_grad(const aqfq_qspec* spec, const void* x, const void* dy, int64_t batch,
                       int64_t rows, int64_t K, const float* scale, const float* tensor_scale,
                       float* dscale, float* dtensor_scale, void* dx, const void* y,
                       void* workspace, size_t workspace_bytes, Problem& p) {
  aqfq_status s = make_problem(spec, batch, rows, K, p);
  if (s != AQFQ_OK) return s;
  if (p.gran == AQFQ_PER_HEAD && p.rows * int64_t(p.cpr) > (int64_t(1) << 24)) return AQFQ_ERR_SHAPE;
  if (elems(p) > 0 && (!x || !dy)) return AQFQ_ERR_NULL;
  if ((s = check_scales(p, scale, tensor_scale)) != AQFQ_OK) return s;
  const bool dyn = p.fmt == AQFQ_NVFP4 && p.mode == AQFQ_SCALE_DYNAMIC_BLOCK;
  if (dyn) {
    if (!dtensor_scale && p.batch > 0) return AQFQ_ERR_NULL;
    if (dscale) return AQFQ_ERR_UNSUPPORTED;
  } else {
    if (!dscale && scale_count(p) > 0) return AQFQ_ERR_NULL;
    if (dtensor_scale) return AQFQ_ERR_UNSUPPORTED;
  }
  if ((s = choose_layout(p, {x, dy, dx, y})) != AQFQ_OK) return s;
  if ((dscale && !aligned(dscale, 4)) || (dtensor_scale && !aligned(dtensor_scale, 4)))
    return AQFQ_ERR_ALIGN;
  if (aqfq::sm_count() <= 0) return AQFQ_ERR_CUDA;  // grids and workspace follow the SM count
  const size_t need = aqfq::grad_workspace_bytes(p);
  if (need > 0) {
    if (!workspace) return AQFQ_ERR_WORKSPACE;
    if (workspace_bytes < need) return AQFQ_ERR_WORKSPACE;
    if (!aligned(workspace, 8)) return AQFQ_ERR_ALIGN;
  }
  return AQFQ_OK;
}

}  // namespace

extern "C" {

aqfq_status aqfq_scale_grad(const aqfq_qspec* spec, const void* x, const void* dy, int64_t batch,
                            int64_t rows, int64_t K, const float* scale,
                            const float* tensor_scale, float* dscale, float* dtensor_scale,
                            void* dx, int accumulate, void* workspace, size_t workspace_bytes,
                            void* stream) {
  Problem p;
  aqfq_status s = check_grad(spec, x, dy, batch, rows, K, scale, tensor_scale, dscale,
                             dtensor_scale, dx, nullptr, workspace, workspace_bytes, p);
  if (s != AQFQ_OK) return s;
  return finish(aqfq::launch_scale_grad(p, x, dy, scale, tensor_scale, dscale, dtensor_scale, dx,
                                        accumulate, static_cast<double*>(workspace),
                                        static_cast<cudaStream_t>(stream)));
}

aqfq_status aqfq_qdq_fwd_grad(const aqfq_qspec* spec, const void* x, const void* dy,
                              int64_t batch, int64_t rows, int64_t K, const float* scale,
                              const float* tensor_scale, void* y, float* dscale,
                              float* dtensor_scale, void* dx, int accumulate, void* workspace,
                              size_t workspace_bytes, void* stream) {
  Problem p;
  if (!spec) return AQFQ_ERR_NULL;
  {
    Problem q;  // y is required whenever there are elements
    const aqfq_status s0 = make_problem(spec, batch, rows, K, q);
    if (s0 != AQFQ_OK) return s0;
    if (!y && elems(q) > 0) return AQFQ_ERR_NULL;
  }
  aqfq_status s = check_grad(spec, x, dy, batch, rows, K, scale, tensor_scale, dscale,
                             dtensor_scale, dx, y, workspace, workspace_bytes, p);
  if (s != AQFQ_OK) return s;
  return finish(aqfq::launch_qdq_fwd_grad(p, x, dy, scale, tensor_scale, y, dscale, dtensor_scale,
                                          dx, accumulate, static_cast<double*>(workspace),
                                          static_cast<cudaStream_t>(stream)));
}

aqfq_status aqfq_observer_minmax(const void* x, int64_t T, int64_t H, int64_t D, float* min_out,
                                 float* max_out, int accumulate, void* stream) {
  if (T < 0 || H < 0 || D < 0 || D % 8 != 0) return AQFQ_ERR_SHAPE;
  const int64_t ce = (D % 16 == 0) ? 16 : 8;
  if (H * (D / ce) > (int64_t(1) << 24)) return AQFQ_ERR_SHAPE;
  if (T > 0 && H * (D / ce) > 0 && T > (int64_t(1) << 40) / (H * (D / ce))) return AQFQ_ERR_SHAPE;
  if ((!x && T * H * D > 0) || ((!min_out || !max_out) && H > 0)) return AQFQ_ERR_NULL;
  if (!aligned(x, 16)) return AQFQ_ERR_ALIGN;
  if (!aligned(min_out, 4) || !aligned(max_out, 4)) return AQFQ_ERR_ALIGN;
  if (aqfq::sm_count() <= 0) return AQFQ_ERR_CUDA;
  const int lay = ce == 8 ? aqfq::L_8 : (aligned(x, 32) ? aqfq::L_32 : aqfq::L_16);
  return finish(aqfq::launch_observer(x, T, H, D, lay, min_out, max_out, accumulate,
                                      static_cast<cudaStream_t>(stream)));
}

aqfq_status aqfq_minmax_scale(const float* min_in, const float* max_in, int64_t H, float qmax,
                              float* scale_out, void* stream) {
  if (H < 0 || !(qmax > 0.0f)) return AQFQ_ERR_SHAPE;
  if ((!min_in || !max_in || !scale_out) && H > 0) return AQFQ_ERR_NULL;
  if (!aligned(min_in, 4) || !aligned(max_in, 4) || !aligned(scale_out, 4)) return AQFQ_ERR_ALIGN;
  return finish(aqfq::launch_minmax_scale(min_in, max_in, H, qmax, scale_out,
                                          static_cast<cudaStream_t>(stream)));
}

aqfq_status aqfq_scale_init(const aqfq_qspec* spec, const void* x, int64_t batch, int64_t rows,
                            int64_t K, float* scale, float* tensor_scale, void* stream) {
  Problem p;
  aqfq_status s = make_problem(spec, batch, rows, K, p);
  if (s != AQFQ_OK) return s;
  if (!x && elems(p) > 0) return AQFQ_ERR_NULL;
  if ((s = check_scales(p, scale, tensor_scale)) != AQFQ_OK) return s;
  if ((s = choose_layout(p, {x})) != AQFQ_OK) return s;
  return finish(aqfq::launch_scale_init(p, x, scale, tensor_scale,
                                        static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
