// dit_internal.h -- host-side interface between the C ABI (dit_api.cu) and
// the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace dit {

enum Op { OP_RGA = 0, OP_MOD = 1, OP_FUSED = 2 };

// Most problems one grouped launch takes (DIT_MAX_GROUP of the C ABI).
constexpr int kMaxGroup = 8;

// Arguments of the flat (full-gate) residual-gate kernel.  Elements
// [0, n_head) and the n_tail elements after the vector body are handled one
// at a time; the body is n_vec vectors of the kernel's width.
struct FlatArgs {
  void* out;
  const void* h;
  const void* u;
  const void* g;
  int64_t n_head;
  int64_t n_vec;
  int64_t n_tail;
};

// Arguments of the row kernels.  Pointers are the tensors of the call; each
// kernel reads only those its operation uses.
struct RowArgs {
  void* out;          // residual gate: out; modulation: out; fused: residual_out
  void* out2;         // fused: modulated_out
  const void* x;      // residual gate / fused: hidden; modulation: x
  const void* u;      // update
  const void* g;      // gate
  const void* sc;     // scale
  const void* sh;     // shift
  int64_t L;          // rows per batch
  int64_t D;          // elements per row
  int64_t rows;       // B * L
  int64_t vstride;    // bytes between batches of a [B, 1, D] operand (D * s when contiguous)
  int64_t nvec;       // vectors of the kernel's width per row
  float eps;
  float d_f;          // D as fp32 (exact: D <= 2^24)
  float inv_d;        // fl(1 / D): the fast statistic's quotient
  int exact;          // the exact statistic (dit_set_statistic) when nonzero
  // grid-stride schedule of the row kernels: groups of rows, never
  // straddling a batch; CTA c takes groups c, c + G, c + 2G, ...
  int64_t gpb;        // groups per batch
  int64_t ngroups;    // B * gpb
  // (the two-warp kernel: step_b = `head`, the first CTAs of a batch, which
  // stride over its rows [0, step_g); the others take one row per team of
  // the rest.  Reused rather than added: a larger struct made the grouped
  // kernel, which holds eight of them, 3.7% slower)
  int64_t step_b;     // G / gpb
  int64_t step_g;     // G % gpb
  const float* qscale;  // E4M3 output: the per-tensor quantisation scale (device)
};

struct DeviceInfo {
  int device;
  int sm_count;
  int smem_optin;  // largest static + dynamic shared memory one CTA may use
};

// The current device's SM count and shared-memory limit, cached per device.
cudaError_t current_device(DeviceInfo* info);
// How many CTAs of `fn` at `block` threads (and `smem` bytes of dynamic
// shared memory) are resident per SM (cached).
int resident_ctas(const DeviceInfo& dev, const void* fn, int block, size_t smem = 0);

// Widest power-of-two access (<= 32 bytes) that divides every address and
// byte pitch in `bits` (the OR of them all).
#ifndef DIT_MAX_ACCESS
#define DIT_MAX_ACCESS 32
#endif
inline int widest_access(uint64_t bits) {
  int vb = DIT_MAX_ACCESS;
  while (vb > 1 && (bits & (uint64_t)(vb - 1))) vb >>= 1;
  return vb;
}

// Launchers, one per operation family (defined in k_*.cu).  dtype is a
// dit_dtype value, vb the access width in bytes.
cudaError_t launch_rga_full(const DeviceInfo& dev, int dtype, void* out,
                            const void* h, const void* u, const void* g,
                            int64_t n, cudaStream_t stream);
cudaError_t launch_rga_bcast(const DeviceInfo& dev, int dtype, int vb,
                             const RowArgs& a, int64_t B, cudaStream_t stream);
cudaError_t launch_modulate(const DeviceInfo& dev, int dtype, int vb,
                            bool mod_full, const RowArgs& a, int64_t B,
                            cudaStream_t stream);
cudaError_t launch_gelu(const DeviceInfo& dev, int dtype, void* out, const void* x,
                        int64_t n, cudaStream_t stream);
cudaError_t launch_fused(const DeviceInfo& dev, int dtype, int vb,
                         bool gate_full, bool mod_full, const RowArgs& a,
                         int64_t B, cudaStream_t stream);
// The modulation / fused op with an E4M3 modulated output (a.qscale set):
// staged rows only (16-byte aligned, at most 8192 16-bit or 4096 fp32
// elements); cudaErrorNotSupported otherwise.
cudaError_t launch_modulate_fp8(const DeviceInfo& dev, int dtype, bool mod_full,
                                const RowArgs& a, int64_t B, cudaStream_t stream);
cudaError_t launch_fused_fp8(const DeviceInfo& dev, int dtype, bool gate_full, bool mod_full,
                             const RowArgs& a, int64_t B, cudaStream_t stream);

// Grouped launches of the staged row kernel: `count` problems of one
// operation, dtype and layout, each with 16-byte aligned rows.  Return
// cudaErrorNotSupported, having launched nothing, when a problem cannot take
// the staged kernel (the caller then launches the problems one by one).
cudaError_t launch_rga_grouped(const DeviceInfo& dev, int dtype, const RowArgs* a,
                               const int64_t* B, int count, cudaStream_t stream);
cudaError_t launch_modulate_grouped(const DeviceInfo& dev, int dtype, bool mod_full,
                                    const RowArgs* a, const int64_t* B, int count,
                                    cudaStream_t stream);
cudaError_t launch_fused_grouped(const DeviceInfo& dev, int dtype, bool gate_full,
                                 bool mod_full, const RowArgs* a, const int64_t* B, int count,
                                 cudaStream_t stream);

// The self-check of one runtime key (dit_selfcheck): nine tensors of a
// [B, L, D] problem in the caller's workspace -- x (hidden), update, gate,
// scale, shift, out, out2, expected, expected2 -- and B * L row statistics.
struct SelfcheckArgs {
  void* t[9];
  float* rstat;
  int64_t D;
  int B, L;
  int dtype;
  int op;  // Op
  bool gate_full, mod_full;
  float eps;
};
// seeded inputs; the plain reference outputs; the count of differing output
// words added to *mismatches (k_selfcheck.cu)
cudaError_t launch_selfcheck_fill(const SelfcheckArgs& a, cudaStream_t s);
cudaError_t launch_selfcheck_reference(const SelfcheckArgs& a, cudaStream_t s);
cudaError_t launch_selfcheck_compare(const SelfcheckArgs& a, unsigned int* mismatches,
                                     cudaStream_t s);

// ---------------------------------------------------------------------------
// compile-time dispatch over (dtype, access width)
// ---------------------------------------------------------------------------
template <class T>
struct TypeTag {
  using type = T;
};
template <int V>
using Width = std::integral_constant<int, V>;

template <class T, class Fn>
cudaError_t dispatch_width(int vb, Fn&& fn) {
  switch (vb) {
    case 32: return fn(TypeTag<T>{}, Width<32>{});
    case 16: return fn(TypeTag<T>{}, Width<16>{});
    case 8:  return fn(TypeTag<T>{}, Width<8>{});
    case 4:  return fn(TypeTag<T>{}, Width<4>{});
    case 2:
      if constexpr (sizeof(T) == 2) return fn(TypeTag<T>{}, Width<2>{});
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <class Fn>
cudaError_t dispatch_dtype_width(int dtype, int vb, Fn&& fn) {
  switch (dtype) {
    case 0: return dispatch_width<__nv_bfloat16>(vb, fn);
    case 1: return dispatch_width<__half>(vb, fn);
    case 2: return dispatch_width<float>(vb, fn);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dit
