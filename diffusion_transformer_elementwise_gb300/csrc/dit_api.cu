// dit_api.cu -- the C ABI of libdit_elementwise.so (include/dit_elementwise.h):
// argument validation, aliasing rules, access-width choice and the per-device
// launch-limit cache.  Every entry point validates on the host, enqueues one
// kernel on the caller's stream and returns; nothing is allocated.
#include <math.h>

#include <map>
#include <mutex>
#include <tuple>

#include "dit_elementwise.h"
#include "dit_internal.h"

namespace dit {

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];  // 0 = not yet queried
int g_smem_optin[kMaxDevices];
std::mutex g_mu;
std::map<std::tuple<int, const void*, int, size_t>, int> g_resident;
}  // namespace

cudaError_t current_device(DeviceInfo* info) {
  int d = -1;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  int c = 0, optin = 0;
  const bool cached = d >= 0 && d < kMaxDevices;
  if (cached) {
    c = __atomic_load_n(&g_sm_count[d], __ATOMIC_ACQUIRE);
    optin = __atomic_load_n(&g_smem_optin[d], __ATOMIC_ACQUIRE);
  }
  if (c == 0 || optin == 0) {
    e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, d);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    if (e != cudaSuccess) return e;
    if (cached) {
      __atomic_store_n(&g_smem_optin[d], optin, __ATOMIC_RELEASE);
      __atomic_store_n(&g_sm_count[d], c, __ATOMIC_RELEASE);
    }
  }
  info->device = d;
  info->sm_count = c > 0 ? c : 1;
  info->smem_optin = optin;
  return cudaSuccess;
}

int resident_ctas(const DeviceInfo& dev, const void* fn, int block, size_t smem) {
  const auto key = std::make_tuple(dev.device, fn, block, smem);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_resident.find(key);
    if (it != g_resident.end()) return it->second;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, block, smem) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();  // the query's own error is not the caller's
    n = 1;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  g_resident[key] = n;
  return n;
}

}  // namespace dit

using dit::DeviceInfo;
using dit::RowArgs;

namespace {

int elem_size(dit_dtype t) { return t == DIT_FP32 ? 4 : 2; }

bool valid_dtype(int t) { return t == DIT_BF16 || t == DIT_FP16 || t == DIT_FP32; }
bool valid_layout(int l) { return l == DIT_FULL || l == DIT_ROW_BCAST; }

// N = B * L * D elements; false on a negative size or overflow of the byte
// count of a tensor.
bool element_count(int64_t B, int64_t L, int64_t D, int es, int64_t* n) {
  if (B < 0 || L < 0 || D < 0) return false;
  int64_t bl, bld, bytes;
  if (__builtin_mul_overflow(B, L, &bl)) return false;
  if (__builtin_mul_overflow(bl, D, &bld)) return false;
  if (__builtin_mul_overflow(bld, (int64_t)es, &bytes)) return false;
  *n = bld;
  return true;
}

struct Span {
  uintptr_t lo, hi;  // [lo, hi) bytes
};
Span span(const void* p, int64_t bytes) {
  return Span{(uintptr_t)p, (uintptr_t)p + (uintptr_t)bytes};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

bool misaligned(const void* p, int es) { return ((uintptr_t)p & (uintptr_t)(es - 1)) != 0; }

dit_status launch_status(cudaError_t e) { return e == cudaSuccess ? DIT_OK : DIT_ERR_LAUNCH; }

}  // namespace

extern "C" {

int dit_abi_version(void) { return DIT_ABI_VERSION; }

const char* dit_status_string(dit_status s) {
  switch (s) {
    case DIT_OK: return "DIT_OK";
    case DIT_ERR_NULL_PTR: return "DIT_ERR_NULL_PTR: a tensor pointer is NULL";
    case DIT_ERR_BAD_SHAPE: return "DIT_ERR_BAD_SHAPE: B, L or D negative, or the size overflows";
    case DIT_ERR_BAD_DTYPE: return "DIT_ERR_BAD_DTYPE: dtype is not bf16, fp16 or fp32";
    case DIT_ERR_BAD_LAYOUT: return "DIT_ERR_BAD_LAYOUT: layout is not full or row-broadcast";
    case DIT_ERR_ALIAS: return "DIT_ERR_ALIAS: an output overlaps another tensor";
    case DIT_ERR_BAD_EPS: return "DIT_ERR_BAD_EPS: eps must be finite and >= 0";
    case DIT_ERR_LAUNCH: return "DIT_ERR_LAUNCH: the CUDA runtime rejected the launch";
    case DIT_ERR_MISALIGNED: return "DIT_ERR_MISALIGNED: a pointer is not aligned to the element size";
    case DIT_ERR_NO_DEVICE: return "DIT_ERR_NO_DEVICE: no current CUDA device";
  }
  return "unknown dit_status";
}

}  // extern "C"

namespace {

// Bytes a [B, 1, D] operand spans with a batch stride of vs elements.
int64_t vector_span(int64_t B, int64_t D, int64_t vs, int es) { return ((B - 1) * vs + D) * es; }

// A stride of vs elements between batches: at least D when B > 1 (any value
// when B == 1, where only one vector is read), and no overflow of the span.
bool valid_vector_stride(int64_t B, int64_t D, int64_t vs, int es) {
  if (B <= 1) return true;
  if (vs < D) return false;
  int64_t t;
  return !__builtin_mul_overflow(B - 1, vs, &t) && !__builtin_mul_overflow(t + D, (int64_t)es, &t);
}

dit_status residual_gate_impl(void* out, const void* hidden, const void* update, const void* gate,
                              int64_t B, int64_t L, int64_t D, dit_dtype dtype,
                              dit_layout gate_layout, int64_t vs, dit_stream_t stream) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(gate_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool full = gate_layout == DIT_FULL;
  if (!full && !valid_vector_stride(B, D, vs, es)) return DIT_ERR_BAD_SHAPE;
  if (n == 0) return DIT_OK;
  if (!out || !hidden || !update || !gate) return DIT_ERR_NULL_PTR;
  if (misaligned(out, es) || misaligned(hidden, es) || misaligned(update, es) ||
      misaligned(gate, es))
    return DIT_ERR_MISALIGNED;
  const int64_t bytes = n * es;
  const Span so = span(out, bytes);
  if (overlaps(so, span(update, bytes)) ||
      overlaps(so, span(gate, full ? bytes : vector_span(B, D, vs, es))) ||
      (out != hidden && overlaps(so, span(hidden, bytes))))
    return DIT_ERR_ALIAS;

  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  cudaStream_t s = (cudaStream_t)stream;
  if (full) return launch_status(dit::launch_rga_full(dev, dtype, out, hidden, update, gate, n, s));

  RowArgs a = {};
  a.out = out;
  a.x = hidden;
  a.u = update;
  a.g = gate;
  a.L = L;
  a.D = D;
  a.rows = B * L;
  a.vstride = (B > 1 ? vs : D) * es;
  const uint64_t bits = (uintptr_t)out | (uintptr_t)hidden | (uintptr_t)update |
                        (uintptr_t)gate | (uint64_t)(D * es) | (uint64_t)a.vstride;
  return launch_status(dit::launch_rga_bcast(dev, dtype, dit::widest_access(bits), a, B, s));
}

dit_status modulate_impl(void* out, const void* x, const void* scale, const void* shift,
                         int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
                         dit_layout mod_layout, int64_t vs, dit_stream_t stream) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(mod_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool full = mod_layout == DIT_FULL;
  if (!full && !valid_vector_stride(B, D, vs, es)) return DIT_ERR_BAD_SHAPE;
  if (!(eps >= 0.0f) || isinf(eps)) return DIT_ERR_BAD_EPS;
  if (n == 0) return DIT_OK;
  if (!out || !x || !scale || !shift) return DIT_ERR_NULL_PTR;
  if (misaligned(out, es) || misaligned(x, es) || misaligned(scale, es) || misaligned(shift, es))
    return DIT_ERR_MISALIGNED;
  const int64_t bytes = n * es;
  const int64_t vbytes = full ? bytes : vector_span(B, D, vs, es);
  const Span so = span(out, bytes);
  if (overlaps(so, span(x, bytes)) || overlaps(so, span(scale, vbytes)) ||
      overlaps(so, span(shift, vbytes)))
    return DIT_ERR_ALIAS;

  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  RowArgs a = {};
  a.out = out;
  a.x = x;
  a.sc = scale;
  a.sh = shift;
  a.L = L;
  a.D = D;
  a.rows = B * L;
  a.vstride = (B > 1 && !full ? vs : D) * es;
  a.eps = eps;
  a.d_f = (float)D;
  a.inv_d = 1.0f / (float)D;
  const uint64_t bits = (uintptr_t)out | (uintptr_t)x | (uintptr_t)scale | (uintptr_t)shift |
                        (uint64_t)(D * es) | (uint64_t)a.vstride;
  return launch_status(dit::launch_modulate(dev, dtype, dit::widest_access(bits), full, a, B,
                                            (cudaStream_t)stream));
}

dit_status fused_impl(void* residual_out, void* modulated_out, const void* hidden,
                      const void* update, const void* gate, const void* scale, const void* shift,
                      int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
                      dit_layout gate_layout, dit_layout mod_layout, int64_t vs,
                      dit_stream_t stream) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(gate_layout) || !valid_layout(mod_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool any_bcast = gate_layout == DIT_ROW_BCAST || mod_layout == DIT_ROW_BCAST;
  if (any_bcast && !valid_vector_stride(B, D, vs, es)) return DIT_ERR_BAD_SHAPE;
  if (!(eps >= 0.0f) || isinf(eps)) return DIT_ERR_BAD_EPS;
  if (n == 0) return DIT_OK;
  if (!residual_out || !modulated_out || !hidden || !update || !gate || !scale || !shift)
    return DIT_ERR_NULL_PTR;
  if (misaligned(residual_out, es) || misaligned(modulated_out, es) || misaligned(hidden, es) ||
      misaligned(update, es) || misaligned(gate, es) || misaligned(scale, es) ||
      misaligned(shift, es))
    return DIT_ERR_MISALIGNED;
  const int64_t bytes = n * es;
  const int64_t vbytes = vector_span(B, D, vs, es);
  const int64_t gbytes = gate_layout == DIT_FULL ? bytes : vbytes;
  const int64_t mbytes = mod_layout == DIT_FULL ? bytes : vbytes;
  const Span sr = span(residual_out, bytes);
  const Span sm = span(modulated_out, bytes);
  const Span inputs[5] = {span(hidden, bytes), span(update, bytes), span(gate, gbytes),
                          span(scale, mbytes), span(shift, mbytes)};
  if (overlaps(sr, sm)) return DIT_ERR_ALIAS;
  for (int i = 0; i < 5; ++i) {
    if (overlaps(sm, inputs[i])) return DIT_ERR_ALIAS;
    if (i == 0 && residual_out == hidden) continue;
    if (overlaps(sr, inputs[i])) return DIT_ERR_ALIAS;
  }

  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  RowArgs a = {};
  a.out = residual_out;
  a.out2 = modulated_out;
  a.x = hidden;
  a.u = update;
  a.g = gate;
  a.sc = scale;
  a.sh = shift;
  a.L = L;
  a.D = D;
  a.rows = B * L;
  a.vstride = (B > 1 && any_bcast ? vs : D) * es;
  a.eps = eps;
  a.d_f = (float)D;
  a.inv_d = 1.0f / (float)D;
  const uint64_t bits = (uintptr_t)residual_out | (uintptr_t)modulated_out | (uintptr_t)hidden |
                        (uintptr_t)update | (uintptr_t)gate | (uintptr_t)scale |
                        (uintptr_t)shift | (uint64_t)(D * es) | (uint64_t)a.vstride;
  return launch_status(dit::launch_fused(dev, dtype, dit::widest_access(bits),
                                         gate_layout == DIT_FULL, mod_layout == DIT_FULL, a, B,
                                         (cudaStream_t)stream));
}

}  // namespace

extern "C" {

dit_status dit_residual_gate_add(void* out, const void* hidden, const void* update,
                                 const void* gate, int64_t B, int64_t L, int64_t D,
                                 dit_dtype dtype, dit_layout gate_layout,
                                 dit_stream_t stream) {
  return residual_gate_impl(out, hidden, update, gate, B, L, D, dtype, gate_layout, D, stream);
}

dit_status dit_rmsnorm_modulate(void* out, const void* x, const void* scale, const void* shift,
                                int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
                                dit_layout mod_layout, dit_stream_t stream) {
  return modulate_impl(out, x, scale, shift, B, L, D, eps, dtype, mod_layout, D, stream);
}

dit_status dit_gate_add_rmsnorm_modulate(void* residual_out, void* modulated_out,
                                         const void* hidden, const void* update,
                                         const void* gate, const void* scale,
                                         const void* shift, int64_t B, int64_t L, int64_t D,
                                         float eps, dit_dtype dtype, dit_layout gate_layout,
                                         dit_layout mod_layout, dit_stream_t stream) {
  return fused_impl(residual_out, modulated_out, hidden, update, gate, scale, shift, B, L, D, eps,
                    dtype, gate_layout, mod_layout, D, stream);
}

dit_status dit_gelu_tanh(void* out, const void* x, int64_t n, dit_dtype dtype,
                         dit_stream_t stream) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  const int es = elem_size(dtype);
  int64_t bytes;
  if (n < 0 || __builtin_mul_overflow(n, (int64_t)es, &bytes)) return DIT_ERR_BAD_SHAPE;
  if (n == 0) return DIT_OK;
  if (!out || !x) return DIT_ERR_NULL_PTR;
  if (misaligned(out, es) || misaligned(x, es)) return DIT_ERR_MISALIGNED;
  if (out != x && overlaps(span(out, bytes), span(x, bytes))) return DIT_ERR_ALIAS;
  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  return launch_status(dit::launch_gelu(dev, dtype, out, x, n, (cudaStream_t)stream));
}

dit_status dit_residual_gate_add_strided(void* out, const void* hidden, const void* update,
                                         const void* gate, int64_t B, int64_t L, int64_t D,
                                         dit_dtype dtype, dit_layout gate_layout,
                                         int64_t vec_stride, dit_stream_t stream) {
  return residual_gate_impl(out, hidden, update, gate, B, L, D, dtype, gate_layout, vec_stride,
                            stream);
}

dit_status dit_rmsnorm_modulate_strided(void* out, const void* x, const void* scale,
                                        const void* shift, int64_t B, int64_t L, int64_t D,
                                        float eps, dit_dtype dtype, dit_layout mod_layout,
                                        int64_t vec_stride, dit_stream_t stream) {
  return modulate_impl(out, x, scale, shift, B, L, D, eps, dtype, mod_layout, vec_stride, stream);
}

dit_status dit_gate_add_rmsnorm_modulate_strided(
    void* residual_out, void* modulated_out, const void* hidden, const void* update,
    const void* gate, const void* scale, const void* shift, int64_t B, int64_t L, int64_t D,
    float eps, dit_dtype dtype, dit_layout gate_layout, dit_layout mod_layout,
    int64_t vec_stride, dit_stream_t stream) {
  return fused_impl(residual_out, modulated_out, hidden, update, gate, scale, shift, B, L, D, eps,
                    dtype, gate_layout, mod_layout, vec_stride, stream);
}

}  // extern "C"
