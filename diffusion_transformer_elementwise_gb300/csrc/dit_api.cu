// dit_api.cu -- the C ABI of libdit_elementwise.so (include/dit_elementwise.h):
// argument validation, aliasing rules, access-width choice and the per-device
// launch-limit cache.  Every entry point validates on the host, enqueues one
// kernel on the caller's stream and returns; nothing is allocated.
#include <math.h>

#include <atomic>
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

// The process's row statistic (dit_set_statistic), read when a call is made.
std::atomic<int> g_statistic{DIT_STATISTIC_FAST};

void set_statistic(RowArgs& a, int64_t D) {
  a.inv_d = 1.0f / (float)D;
  a.exact = g_statistic.load(std::memory_order_relaxed) == DIT_STATISTIC_EXACT;
}

}  // namespace

extern "C" {

int dit_abi_version(void) { return DIT_ABI_VERSION; }

dit_status dit_set_statistic(dit_statistic statistic) {
  if (statistic != DIT_STATISTIC_FAST && statistic != DIT_STATISTIC_EXACT)
    return DIT_ERR_BAD_STATISTIC;
  g_statistic.store((int)statistic, std::memory_order_relaxed);
  return DIT_OK;
}

dit_statistic dit_get_statistic(void) {
  return (dit_statistic)g_statistic.load(std::memory_order_relaxed);
}

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
    case DIT_ERR_BAD_OP:
      return "DIT_ERR_BAD_OP: op is not a dit_op value, or count is outside [0, DIT_MAX_GROUP]";
    case DIT_ERR_WORKSPACE:
      return "DIT_ERR_WORKSPACE: workspace NULL, too small or not 256-byte aligned";
    case DIT_ERR_BAD_STATISTIC:
      return "DIT_ERR_BAD_STATISTIC: not a dit_statistic value";
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

// The longest row the modulating operations take: D is exact in fp32 and the
// exact path's 64-bit digit totals cannot overflow.
constexpr int64_t kMaxStatisticRow = int64_t(1) << 24;

// A validated call of one operation: its kernel arguments, its access width
// and the byte spans it writes and reads (for the aliasing checks of grouped
// calls).
struct Prepared {
  int op;
  bool empty;
  int64_t B;
  int64_t n;  // B * L * D
  RowArgs a;
  int vb;  // widest access dividing every row pointer, the pitch and the stride
  bool gate_full, mod_full;
  Span writes[2];
  int nwrites;
  Span reads[5];
  int nreads;
};

dit_status prepare_rga(void* out, const void* hidden, const void* update, const void* gate,
                       int64_t B, int64_t L, int64_t D, dit_dtype dtype, dit_layout gate_layout,
                       int64_t vs, Prepared* p) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(gate_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool full = gate_layout == DIT_FULL;
  if (!full && !valid_vector_stride(B, D, vs, es)) return DIT_ERR_BAD_SHAPE;
  *p = Prepared{};
  p->op = dit::OP_RGA;
  p->empty = n == 0;
  if (p->empty) return DIT_OK;
  if (!out || !hidden || !update || !gate) return DIT_ERR_NULL_PTR;
  if (misaligned(out, es) || misaligned(hidden, es) || misaligned(update, es) ||
      misaligned(gate, es))
    return DIT_ERR_MISALIGNED;
  const int64_t bytes = n * es;
  const Span so = span(out, bytes);
  const Span sg = span(gate, full ? bytes : vector_span(B, D, vs, es));
  if (overlaps(so, span(update, bytes)) || overlaps(so, sg) ||
      (out != hidden && overlaps(so, span(hidden, bytes))))
    return DIT_ERR_ALIAS;

  p->B = B;
  p->n = n;
  p->gate_full = full;
  RowArgs& a = p->a;
  a.out = out;
  a.x = hidden;
  a.u = update;
  a.g = gate;
  a.L = L;
  a.D = D;
  a.rows = B * L;
  a.vstride = (B > 1 && !full ? vs : D) * es;
  const uint64_t bits = (uintptr_t)out | (uintptr_t)hidden | (uintptr_t)update |
                        (uintptr_t)gate | (uint64_t)(D * es) | (uint64_t)a.vstride;
  p->vb = dit::widest_access(bits);
  p->writes[0] = so;
  p->nwrites = 1;
  p->reads[0] = span(hidden, bytes);
  p->reads[1] = span(update, bytes);
  p->reads[2] = sg;
  p->nreads = 3;
  return DIT_OK;
}

dit_status prepare_modulate(void* out, const void* x, const void* scale, const void* shift,
                            int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
                            dit_layout mod_layout, int64_t vs, Prepared* p) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(mod_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool full = mod_layout == DIT_FULL;
  if (!full && !valid_vector_stride(B, D, vs, es)) return DIT_ERR_BAD_SHAPE;
  if (D > kMaxStatisticRow) return DIT_ERR_BAD_SHAPE;
  if (!(eps >= 0.0f) || isinf(eps)) return DIT_ERR_BAD_EPS;
  *p = Prepared{};
  p->op = dit::OP_MOD;
  p->empty = n == 0;
  if (p->empty) return DIT_OK;
  if (!out || !x || !scale || !shift) return DIT_ERR_NULL_PTR;
  if (misaligned(out, es) || misaligned(x, es) || misaligned(scale, es) || misaligned(shift, es))
    return DIT_ERR_MISALIGNED;
  const int64_t bytes = n * es;
  const int64_t vbytes = full ? bytes : vector_span(B, D, vs, es);
  const Span so = span(out, bytes);
  if (overlaps(so, span(x, bytes)) || overlaps(so, span(scale, vbytes)) ||
      overlaps(so, span(shift, vbytes)))
    return DIT_ERR_ALIAS;

  p->B = B;
  p->n = n;
  p->mod_full = full;
  RowArgs& a = p->a;
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
  set_statistic(a, D);
  const uint64_t bits = (uintptr_t)out | (uintptr_t)x | (uintptr_t)scale | (uintptr_t)shift |
                        (uint64_t)(D * es) | (uint64_t)a.vstride;
  p->vb = dit::widest_access(bits);
  p->writes[0] = so;
  p->nwrites = 1;
  p->reads[0] = span(x, bytes);
  p->reads[1] = span(scale, vbytes);
  p->reads[2] = span(shift, vbytes);
  p->nreads = 3;
  return DIT_OK;
}

dit_status prepare_fused(void* residual_out, void* modulated_out, const void* hidden,
                         const void* update, const void* gate, const void* scale,
                         const void* shift, int64_t B, int64_t L, int64_t D, float eps,
                         dit_dtype dtype, dit_layout gate_layout, dit_layout mod_layout,
                         int64_t vs, Prepared* p) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(gate_layout) || !valid_layout(mod_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool any_bcast = gate_layout == DIT_ROW_BCAST || mod_layout == DIT_ROW_BCAST;
  if (any_bcast && !valid_vector_stride(B, D, vs, es)) return DIT_ERR_BAD_SHAPE;
  if (D > kMaxStatisticRow) return DIT_ERR_BAD_SHAPE;
  if (!(eps >= 0.0f) || isinf(eps)) return DIT_ERR_BAD_EPS;
  *p = Prepared{};
  p->op = dit::OP_FUSED;
  p->empty = n == 0;
  if (p->empty) return DIT_OK;
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

  p->B = B;
  p->n = n;
  p->gate_full = gate_layout == DIT_FULL;
  p->mod_full = mod_layout == DIT_FULL;
  RowArgs& a = p->a;
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
  set_statistic(a, D);
  const uint64_t bits = (uintptr_t)residual_out | (uintptr_t)modulated_out | (uintptr_t)hidden |
                        (uintptr_t)update | (uintptr_t)gate | (uintptr_t)scale |
                        (uintptr_t)shift | (uint64_t)(D * es) | (uint64_t)a.vstride;
  p->vb = dit::widest_access(bits);
  p->writes[0] = sr;
  p->writes[1] = sm;
  p->nwrites = 2;
  for (int i = 0; i < 5; ++i) p->reads[i] = inputs[i];
  p->nreads = 5;
  return DIT_OK;
}

// One kernel for one prepared, non-empty call.
cudaError_t launch_one(const DeviceInfo& dev, int dtype, const Prepared& p, cudaStream_t s) {
  switch (p.op) {
    case dit::OP_RGA:
      if (p.gate_full)
        return dit::launch_rga_full(dev, dtype, p.a.out, p.a.x, p.a.u, p.a.g, p.n, s);
      return dit::launch_rga_bcast(dev, dtype, p.vb, p.a, p.B, s);
    case dit::OP_MOD:
      return dit::launch_modulate(dev, dtype, p.vb, p.mod_full, p.a, p.B, s);
    default:
      return dit::launch_fused(dev, dtype, p.vb, p.gate_full, p.mod_full, p.a, p.B, s);
  }
}

dit_status run_one(dit_status st, int dtype, const Prepared& p, dit_stream_t stream) {
  if (st != DIT_OK || p.empty) return st;
  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  return launch_status(launch_one(dev, dtype, p, (cudaStream_t)stream));
}

dit_status residual_gate_impl(void* out, const void* hidden, const void* update, const void* gate,
                              int64_t B, int64_t L, int64_t D, dit_dtype dtype,
                              dit_layout gate_layout, int64_t vs, dit_stream_t stream) {
  Prepared p;
  const dit_status st = prepare_rga(out, hidden, update, gate, B, L, D, dtype, gate_layout, vs, &p);
  return run_one(st, dtype, p, stream);
}

dit_status modulate_impl(void* out, const void* x, const void* scale, const void* shift,
                         int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
                         dit_layout mod_layout, int64_t vs, dit_stream_t stream) {
  Prepared p;
  const dit_status st =
      prepare_modulate(out, x, scale, shift, B, L, D, eps, dtype, mod_layout, vs, &p);
  return run_one(st, dtype, p, stream);
}

dit_status fused_impl(void* residual_out, void* modulated_out, const void* hidden,
                      const void* update, const void* gate, const void* scale, const void* shift,
                      int64_t B, int64_t L, int64_t D, float eps, dit_dtype dtype,
                      dit_layout gate_layout, dit_layout mod_layout, int64_t vs,
                      dit_stream_t stream) {
  Prepared p;
  const dit_status st = prepare_fused(residual_out, modulated_out, hidden, update, gate, scale,
                                      shift, B, L, D, eps, dtype, gate_layout, mod_layout, vs, &p);
  return run_one(st, dtype, p, stream);
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

dit_status dit_grouped(dit_op op, const dit_problem* problems, int count, float eps,
                       dit_dtype dtype, dit_layout gate_layout, dit_layout mod_layout,
                       dit_stream_t stream) {
  if (op != DIT_OP_RESIDUAL_GATE && op != DIT_OP_RMSNORM_MODULATE &&
      op != DIT_OP_GATE_ADD_RMSNORM_MODULATE)
    return DIT_ERR_BAD_OP;
  if (count < 0 || count > DIT_MAX_GROUP) return DIT_ERR_BAD_OP;
  if (count > 0 && !problems) return DIT_ERR_NULL_PTR;
  Prepared prep[DIT_MAX_GROUP];
  for (int i = 0; i < count; ++i) {
    const dit_problem& q = problems[i];
    dit_status st;
    if (op == DIT_OP_RESIDUAL_GATE)
      st = prepare_rga(q.out, q.x, q.update, q.gate, q.B, q.L, q.D, dtype, gate_layout,
                       q.vec_stride, &prep[i]);
    else if (op == DIT_OP_RMSNORM_MODULATE)
      st = prepare_modulate(q.out, q.x, q.scale, q.shift, q.B, q.L, q.D, eps, dtype, mod_layout,
                            q.vec_stride, &prep[i]);
    else
      st = prepare_fused(q.out, q.out2, q.x, q.update, q.gate, q.scale, q.shift, q.B, q.L, q.D,
                         eps, dtype, gate_layout, mod_layout, q.vec_stride, &prep[i]);
    if (st != DIT_OK) return st;
  }
  // the problems run concurrently: none may write what another reads or writes
  for (int i = 0; i < count; ++i) {
    if (prep[i].empty) continue;
    for (int j = 0; j < count; ++j) {
      if (j == i || prep[j].empty) continue;
      for (int w = 0; w < prep[i].nwrites; ++w) {
        for (int k = 0; k < prep[j].nwrites; ++k)
          if (overlaps(prep[i].writes[w], prep[j].writes[k])) return DIT_ERR_ALIAS;
        for (int k = 0; k < prep[j].nreads; ++k)
          if (overlaps(prep[i].writes[w], prep[j].reads[k])) return DIT_ERR_ALIAS;
      }
    }
  }
  int live[DIT_MAX_GROUP];
  int nlive = 0;
  for (int i = 0; i < count; ++i)
    if (!prep[i].empty) live[nlive++] = i;
  if (nlive == 0) return DIT_OK;

  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  cudaStream_t s = (cudaStream_t)stream;
  const bool rows_op = !(op == DIT_OP_RESIDUAL_GATE && gate_layout == DIT_FULL);
  bool staged = nlive > 1 && rows_op;
  for (int i = 0; i < nlive; ++i) staged = staged && prep[live[i]].vb >= 16;
  if (staged) {
    RowArgs a[DIT_MAX_GROUP];
    int64_t B[DIT_MAX_GROUP];
    for (int i = 0; i < nlive; ++i) {
      a[i] = prep[live[i]].a;
      B[i] = prep[live[i]].B;
    }
    cudaError_t e;
    if (op == DIT_OP_RESIDUAL_GATE)
      e = dit::launch_rga_grouped(dev, dtype, a, B, nlive, s);
    else if (op == DIT_OP_RMSNORM_MODULATE)
      e = dit::launch_modulate_grouped(dev, dtype, mod_layout == DIT_FULL, a, B, nlive, s);
    else
      e = dit::launch_fused_grouped(dev, dtype, gate_layout == DIT_FULL, mod_layout == DIT_FULL,
                                    a, B, nlive, s);
    if (e != cudaErrorNotSupported) return launch_status(e);
  }
  for (int i = 0; i < nlive; ++i) {
    const cudaError_t e = launch_one(dev, dtype, prep[live[i]], s);
    if (e != cudaSuccess) return DIT_ERR_LAUNCH;
  }
  return DIT_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// self-check of one runtime key
// ---------------------------------------------------------------------------

namespace {
constexpr int kCheckB = 2, kCheckL = 7;  // rows: 7 per batch (ragged for 4-row groups)
constexpr int64_t kCheckAlign = 256;

bool valid_op(int op) {
  return op == DIT_OP_RESIDUAL_GATE || op == DIT_OP_RMSNORM_MODULATE ||
         op == DIT_OP_GATE_ADD_RMSNORM_MODULATE;
}

// bytes of one workspace tensor (N = 14 * D elements, rounded up to 256);
// -1 on overflow or a bad size
int64_t check_slot_bytes(dit_dtype dtype, int64_t D) {
  if (D <= 0 || !valid_dtype(dtype)) return -1;
  int64_t n;
  if (!element_count(kCheckB, kCheckL, D, elem_size(dtype), &n)) return -1;
  const int64_t bytes = n * elem_size(dtype);
  if (bytes > ((int64_t)1 << 40)) return -1;
  return (bytes + kCheckAlign - 1) / kCheckAlign * kCheckAlign;
}
}  // namespace

extern "C" {

int64_t dit_selfcheck_workspace_bytes(dit_op op, dit_dtype dtype, int64_t D) {
  if (!valid_op(op)) return -1;
  const int64_t slot = check_slot_bytes(dtype, D);
  if (slot < 0) return -1;
  return 9 * slot + kCheckAlign;  // nine tensors, then the row statistics
}

dit_status dit_selfcheck(dit_op op, dit_dtype dtype, dit_layout gate_layout,
                         dit_layout mod_layout, int64_t D, void* workspace,
                         int64_t workspace_bytes, unsigned int* mismatches,
                         dit_stream_t stream) {
  if (!valid_op(op)) return DIT_ERR_BAD_OP;
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(gate_layout) || !valid_layout(mod_layout)) return DIT_ERR_BAD_LAYOUT;
  const int64_t slot = check_slot_bytes(dtype, D);
  if (slot < 0) return DIT_ERR_BAD_SHAPE;
  if (!mismatches) return DIT_ERR_NULL_PTR;
  if (((uintptr_t)mismatches & 3) != 0) return DIT_ERR_MISALIGNED;
  if (!workspace || ((uintptr_t)workspace & (uintptr_t)(kCheckAlign - 1)) != 0 ||
      workspace_bytes < 9 * slot + kCheckAlign)
    return DIT_ERR_WORKSPACE;
  const Span sw = span(workspace, 9 * slot + kCheckAlign);
  if (overlaps(sw, span(mismatches, 4))) return DIT_ERR_ALIAS;

  dit::SelfcheckArgs a = {};
  for (int i = 0; i < 9; ++i) a.t[i] = (char*)workspace + i * slot;
  a.rstat = (float*)((char*)workspace + 9 * slot);
  a.D = D;
  a.B = kCheckB;
  a.L = kCheckL;
  a.dtype = dtype;
  a.eps = 0.75f;
  a.gate_full = gate_layout == DIT_FULL;
  a.mod_full = mod_layout == DIT_FULL;

  // the operation through the public call's own validation
  Prepared p;
  dit_status st;
  if (op == DIT_OP_RESIDUAL_GATE) {
    a.op = dit::OP_RGA;
    a.mod_full = false;
    st = prepare_rga(a.t[5], a.t[0], a.t[1], a.t[2], kCheckB, kCheckL, D, dtype, gate_layout, D,
                     &p);
  } else if (op == DIT_OP_RMSNORM_MODULATE) {
    a.op = dit::OP_MOD;
    a.gate_full = false;
    st = prepare_modulate(a.t[5], a.t[0], a.t[3], a.t[4], kCheckB, kCheckL, D, a.eps, dtype,
                          mod_layout, D, &p);
  } else {
    a.op = dit::OP_FUSED;
    st = prepare_fused(a.t[5], a.t[6], a.t[0], a.t[1], a.t[2], a.t[3], a.t[4], kCheckB, kCheckL,
                       D, a.eps, dtype, gate_layout, mod_layout, D, &p);
  }
  if (st != DIT_OK) return st;

  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(mismatches, 0, sizeof(unsigned int), s) != cudaSuccess) {
    (void)cudaGetLastError();
    return DIT_ERR_LAUNCH;
  }
  cudaError_t e = dit::launch_selfcheck_fill(a, s);
  if (e == cudaSuccess) e = launch_one(dev, dtype, p, s);
  if (e == cudaSuccess) e = dit::launch_selfcheck_reference(a, s);
  if (e == cudaSuccess) e = dit::launch_selfcheck_compare(a, mismatches, s);
  return launch_status(e);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// modulated output in OCP E4M3
// ---------------------------------------------------------------------------

namespace {

// Shape and alignment rules of the E4M3-output calls: the staged row kernel
// only -- 16-byte aligned inputs, rows and vector strides of a multiple of
// 16 bytes, rows of at most 16 KB; the E4M3 output aligned to the bytes of
// its per-granule store (8 for 16-bit inputs, 4 for fp32).
dit_status fp8_rules(int64_t D, int es, int64_t vs_bytes, const void* out8,
                     const void* const* inputs, int ninputs) {
  if (D * es > 16384) return DIT_ERR_BAD_SHAPE;
  if ((D * es) % 16 != 0 || vs_bytes % 16 != 0) return DIT_ERR_MISALIGNED;
  for (int i = 0; i < ninputs; ++i)
    if (((uintptr_t)inputs[i] & 15) != 0) return DIT_ERR_MISALIGNED;
  if (((uintptr_t)out8 & (uintptr_t)(16 / es - 1)) != 0) return DIT_ERR_MISALIGNED;
  return DIT_OK;
}

}  // namespace

extern "C" {

dit_status dit_rmsnorm_modulate_fp8(void* out, const void* x, const void* scale,
                                    const void* shift, int64_t B, int64_t L, int64_t D,
                                    float eps, dit_dtype dtype, dit_layout mod_layout,
                                    int64_t vec_stride, const float* quant_scale,
                                    dit_stream_t stream) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(mod_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool full = mod_layout == DIT_FULL;
  if (!full && !valid_vector_stride(B, D, vec_stride, es)) return DIT_ERR_BAD_SHAPE;
  if (!(eps >= 0.0f) || isinf(eps)) return DIT_ERR_BAD_EPS;
  if (n == 0) return DIT_OK;
  if (!out || !x || !scale || !shift || !quant_scale) return DIT_ERR_NULL_PTR;
  const int64_t vs = B > 1 && !full ? vec_stride : D;
  const void* ins[3] = {x, scale, shift};
  const dit_status rule = fp8_rules(D, es, vs * es, out, ins, 3);
  if (rule != DIT_OK) return rule;
  if (((uintptr_t)quant_scale & 3) != 0) return DIT_ERR_MISALIGNED;
  const int64_t bytes = n * es;
  const int64_t vbytes = full ? bytes : vector_span(B, D, vs, es);
  const Span so = span(out, n);  // one byte per element
  if (overlaps(so, span(x, bytes)) || overlaps(so, span(scale, vbytes)) ||
      overlaps(so, span(shift, vbytes)) || overlaps(so, span(quant_scale, 4)))
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
  a.vstride = vs * es;
  a.eps = eps;
  a.d_f = (float)D;
  set_statistic(a, D);
  a.qscale = quant_scale;
  const cudaError_t e = dit::launch_modulate_fp8(dev, dtype, full, a, B, (cudaStream_t)stream);
  return e == cudaErrorNotSupported ? DIT_ERR_BAD_SHAPE : launch_status(e);
}

dit_status dit_gate_add_rmsnorm_modulate_fp8(
    void* residual_out, void* out, const void* hidden, const void* update, const void* gate,
    const void* scale, const void* shift, int64_t B, int64_t L, int64_t D, float eps,
    dit_dtype dtype, dit_layout gate_layout, dit_layout mod_layout, int64_t vec_stride,
    const float* quant_scale, dit_stream_t stream) {
  if (!valid_dtype(dtype)) return DIT_ERR_BAD_DTYPE;
  if (!valid_layout(gate_layout) || !valid_layout(mod_layout)) return DIT_ERR_BAD_LAYOUT;
  const int es = elem_size(dtype);
  int64_t n;
  if (!element_count(B, L, D, es, &n)) return DIT_ERR_BAD_SHAPE;
  const bool any_bcast = gate_layout == DIT_ROW_BCAST || mod_layout == DIT_ROW_BCAST;
  if (any_bcast && !valid_vector_stride(B, D, vec_stride, es)) return DIT_ERR_BAD_SHAPE;
  if (!(eps >= 0.0f) || isinf(eps)) return DIT_ERR_BAD_EPS;
  if (n == 0) return DIT_OK;
  if (!residual_out || !out || !hidden || !update || !gate || !scale || !shift || !quant_scale)
    return DIT_ERR_NULL_PTR;
  const int64_t vs = B > 1 && any_bcast ? vec_stride : D;
  const void* ins[6] = {residual_out, hidden, update, gate, scale, shift};
  const dit_status rule = fp8_rules(D, es, vs * es, out, ins, 6);
  if (rule != DIT_OK) return rule;
  if (((uintptr_t)quant_scale & 3) != 0) return DIT_ERR_MISALIGNED;
  const int64_t bytes = n * es;
  const int64_t vbytes = vector_span(B, D, vs, es);
  const Span sr = span(residual_out, bytes);
  const Span sq = span(out, n);
  const Span inputs[6] = {span(hidden, bytes),
                          span(update, bytes),
                          span(gate, gate_layout == DIT_FULL ? bytes : vbytes),
                          span(scale, mod_layout == DIT_FULL ? bytes : vbytes),
                          span(shift, mod_layout == DIT_FULL ? bytes : vbytes),
                          span(quant_scale, 4)};
  if (overlaps(sr, sq)) return DIT_ERR_ALIAS;
  for (int i = 0; i < 6; ++i) {
    if (overlaps(sq, inputs[i])) return DIT_ERR_ALIAS;
    if (i == 0 && residual_out == hidden) continue;
    if (overlaps(sr, inputs[i])) return DIT_ERR_ALIAS;
  }

  DeviceInfo dev;
  if (dit::current_device(&dev) != cudaSuccess) return DIT_ERR_NO_DEVICE;
  RowArgs a = {};
  a.out = residual_out;
  a.out2 = out;
  a.x = hidden;
  a.u = update;
  a.g = gate;
  a.sc = scale;
  a.sh = shift;
  a.L = L;
  a.D = D;
  a.rows = B * L;
  a.vstride = vs * es;
  a.eps = eps;
  a.d_f = (float)D;
  set_statistic(a, D);
  a.qscale = quant_scale;
  const cudaError_t e = dit::launch_fused_fp8(dev, dtype, gate_layout == DIT_FULL,
                                              mod_layout == DIT_FULL, a, B, (cudaStream_t)stream);
  return e == cudaErrorNotSupported ? DIT_ERR_BAD_SHAPE : launch_status(e);
}

}  // extern "C"
