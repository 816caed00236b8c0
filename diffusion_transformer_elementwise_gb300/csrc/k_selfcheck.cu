// k_selfcheck.cu -- the device side of dit_selfcheck: seeded inputs, a plain
// reference and a word-by-word comparison.
//
// The pages' runtime guard checks each runtime key of the pointwise fusions
// bit for bit on its first use, and falls back to the model's own math on a
// mismatch (vllm-omni PR #7350, "[Kernel] Enable LTX DiffVAE fusions on SM100
// and SM103", section Purpose).  Here there is no fallback: a key is (operation,
// dtype, layouts, row width D); the check runs the library's own launch path
// for that key on a [2, 7, D] problem whose every output has one correct
// value, computes that value with the plain kernels below, and counts the
// output words that differ.
//
// One correct value: the residual gate is defined to the bit (fp32 multiply,
// fp32 add, one rounding).  The modulation's statistic is not (its sum of
// squares may be taken in any order), so the inputs make it exact: every x
// is +-1/2, the mean of squares is exactly 1/4 in any order, eps = 3/4, and
// r = 1/sqrt(1/4 + 3/4) = 1 on any correct path.  For the fused op the
// residual is built to be +-1/2: update = +-1/4, gate in {+-1/4, +-1/2, +-1,
// +-2}, hidden = target - update * gate, all exact in every dtype.
//
// The reference kernels are deliberately plain: one thread per element (one
// per row for the statistic, summing in index order), the dtype conversions
// of cuda_bf16.h / cuda_fp16.h, and none of the production kernels' helpers.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dit_internal.h"

namespace dit {

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  // SplitMix64 finaliser (Steele, Lea, Flood 2014)
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t draw_bits(int tensor, int64_t i) {
  return mix64(((uint64_t)tensor << 48) ^ (uint64_t)i ^ 0x5E1FC4EC0000ull);
}
// uniform in [lo, hi) from the top 24 bits
__device__ __forceinline__ float draw_uniform(int tensor, int64_t i, float lo, float hi) {
  const float u = (float)(draw_bits(tensor, i) >> 40) * (1.0f / 16777216.0f);
  return lo + (hi - lo) * u;
}

template <class T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }

template <class T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }

enum { kX = 0, kU = 1, kG = 2, kSc = 3, kSh = 4, kOut = 5, kOut2 = 6, kExp = 7, kExp2 = 8 };

// gate of the fused op's inputs: one of +-1/4, +-1/2, +-1, +-2
__device__ __forceinline__ float fused_gate(int64_t gi) {
  const uint64_t b = draw_bits(kG, gi);
  const float mag = (float)(1 << (b & 3)) * 0.25f;
  return (b & 4) ? -mag : mag;
}

template <class T>
__global__ void selfcheck_fill(SelfcheckArgs a) {
  T* x = (T*)a.t[kX];
  T* u = (T*)a.t[kU];
  T* g = (T*)a.t[kG];
  T* sc = (T*)a.t[kSc];
  T* sh = (T*)a.t[kSh];
  const int64_t n = (int64_t)a.B * a.L * a.D;
  const int64_t nvec = (int64_t)a.B * a.D;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t row = i / a.D, d = i - row * a.D, b = row / a.L;
    const int64_t gi = a.gate_full ? i : b * a.D + d;
    if (a.op == OP_RGA) {
      x[i] = from_f<T>(draw_uniform(kX, i, -4.0f, 4.0f));
      u[i] = from_f<T>(draw_uniform(kU, i, -4.0f, 4.0f));
    } else if (a.op == OP_MOD) {
      x[i] = from_f<T>((draw_bits(kX, i) & 1) ? 0.5f : -0.5f);
    } else {
      const float target = (draw_bits(kX, i) & 1) ? 0.5f : -0.5f;
      const float uv = (draw_bits(kU, i) & 1) ? 0.25f : -0.25f;
      u[i] = from_f<T>(uv);
      x[i] = from_f<T>(target - uv * fused_gate(gi));  // exact: dyadic with few bits
    }
    // a [B, 1, D] operand has B * D elements, written by the first B * D threads
    if (a.op != OP_MOD && (a.gate_full || i < nvec))
      g[i] = from_f<T>(a.op == OP_RGA ? draw_uniform(kG, i, -1.0f, 1.0f) : fused_gate(i));
    if (a.op != OP_RGA && (a.mod_full || i < nvec)) {
      sc[i] = from_f<T>(draw_uniform(kSc, i, -1.0f, 1.0f));
      sh[i] = from_f<T>(draw_uniform(kSh, i, -1.0f, 1.0f));
    }
  }
}

// expected residual: rnd(fl(h + fl(u * g))), one thread per element
template <class T>
__global__ void selfcheck_ref_residual(SelfcheckArgs a) {
  const T* h = (const T*)a.t[kX];
  const T* u = (const T*)a.t[kU];
  const T* g = (const T*)a.t[kG];
  T* e = (T*)a.t[kExp];
  const int64_t n = (int64_t)a.B * a.L * a.D;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t row = i / a.D, d = i - row * a.D, b = row / a.L;
    const float gv = to_f<T>(g[a.gate_full ? i : b * a.D + d]);
    e[i] = from_f<T>(__fadd_rn(to_f<T>(h[i]), __fmul_rn(to_f<T>(u[i]), gv)));
  }
}

// per-row statistic r = 1 / sqrt(mean(x^2) + eps), summed in index order
// (exact for the self-check's inputs), one thread per row
template <class T>
__global__ void selfcheck_ref_stat(SelfcheckArgs a) {
  const T* x = (const T*)a.t[a.op == OP_FUSED ? kExp : kX];
  const int64_t rows = (int64_t)a.B * a.L;
  const int64_t r0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r0 >= rows) return;
  float s = 0.0f;
  for (int64_t d = 0; d < a.D; ++d) {
    const float v = to_f<T>(x[r0 * a.D + d]);
    s = __fadd_rn(s, __fmul_rn(v, v));
  }
  const float ms = __fdiv_rn(s, (float)a.D);
  a.rstat[r0] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
}

// expected modulation: rnd(fl(fl(fl(x * r) * fl(1 + scale)) + shift))
template <class T>
__global__ void selfcheck_ref_modulate(SelfcheckArgs a) {
  const T* x = (const T*)a.t[a.op == OP_FUSED ? kExp : kX];
  const T* sc = (const T*)a.t[kSc];
  const T* sh = (const T*)a.t[kSh];
  T* e = (T*)a.t[a.op == OP_FUSED ? kExp2 : kExp];
  const int64_t n = (int64_t)a.B * a.L * a.D;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t row = i / a.D, d = i - row * a.D, b = row / a.L;
    const int64_t vi = a.mod_full ? i : b * a.D + d;
    const float nrm = __fmul_rn(to_f<T>(x[i]), a.rstat[row]);
    const float one = __fadd_rn(1.0f, to_f<T>(sc[vi]));
    e[i] = from_f<T>(__fadd_rn(__fmul_rn(nrm, one), to_f<T>(sh[vi])));
  }
}

// count differing output words (out vs expected; for the fused op also
// out2 vs expected2) into *mismatches
template <class W>
__global__ void selfcheck_compare(SelfcheckArgs a, unsigned int* mismatches) {
  const W* o = (const W*)a.t[kOut];
  const W* e = (const W*)a.t[kExp];
  const W* o2 = (const W*)a.t[kOut2];
  const W* e2 = (const W*)a.t[kExp2];
  const int64_t n = (int64_t)a.B * a.L * a.D;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  unsigned int bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    bad += o[i] != e[i];
    if (a.op == OP_FUSED) bad += o2[i] != e2[i];
  }
  if (bad) atomicAdd(mismatches, bad);
}

template <class Fn>
cudaError_t by_dtype(int dtype, Fn&& fn) {
  switch (dtype) {
    case 0: return fn(TypeTag<__nv_bfloat16>{});
    case 1: return fn(TypeTag<__half>{});
    case 2: return fn(TypeTag<float>{});
    default: return cudaErrorInvalidValue;
  }
}

constexpr int kBlock = 256;

unsigned grid_for(int64_t n) {
  int64_t g = (n + kBlock - 1) / kBlock;
  if (g > 1024) g = 1024;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_selfcheck_fill(const SelfcheckArgs& a, cudaStream_t s) {
  const int64_t n = (int64_t)a.B * a.L * a.D;
  return by_dtype(a.dtype, [&](auto tt) -> cudaError_t {
    using T = typename decltype(tt)::type;
    selfcheck_fill<T><<<grid_for(n), kBlock, 0, s>>>(a);
    return cudaGetLastError();
  });
}

cudaError_t launch_selfcheck_reference(const SelfcheckArgs& a, cudaStream_t s) {
  const int64_t n = (int64_t)a.B * a.L * a.D;
  const int64_t rows = (int64_t)a.B * a.L;
  return by_dtype(a.dtype, [&](auto tt) -> cudaError_t {
    using T = typename decltype(tt)::type;
    if (a.op != OP_MOD) selfcheck_ref_residual<T><<<grid_for(n), kBlock, 0, s>>>(a);
    if (a.op != OP_RGA) {
      selfcheck_ref_stat<T><<<(unsigned)((rows + 63) / 64), 64, 0, s>>>(a);
      selfcheck_ref_modulate<T><<<grid_for(n), kBlock, 0, s>>>(a);
    }
    return cudaGetLastError();
  });
}

cudaError_t launch_selfcheck_compare(const SelfcheckArgs& a, unsigned int* mismatches,
                                     cudaStream_t s) {
  const int64_t n = (int64_t)a.B * a.L * a.D;
  if (a.dtype == 2)
    selfcheck_compare<uint32_t><<<grid_for(n), kBlock, 0, s>>>(a, mismatches);
  else
    selfcheck_compare<uint16_t><<<grid_for(n), kBlock, 0, s>>>(a, mismatches);
  return cudaGetLastError();
}

}  // namespace dit
