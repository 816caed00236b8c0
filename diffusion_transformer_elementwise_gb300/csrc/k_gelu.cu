// k_gelu.cu -- tanh-approximated GELU, elementwise, on GB300.
//
// gelu(x) = 0.5 * x * (1 + tanh(z)),  z = sqrt(2/pi) * (x + 0.044715 * x^3):
// the activation of the LTX-2 feed-forward (prhub summary of sglang PR #34172,
// "implementation breakdown" item 3: LTX2FeedForward's tanh-GELU after
// proj_in).  Since 1 + tanh(z) = 2 / (1 + e^(-2z)), the value is
//
//   z >= 0:  x * q             q = 1 / (1 + e^(-2|z|))
//   z <  0:  x * q * e^(-2|z|)
//
// with e^(-2|z|) in (0, 1]: no cancellation and no overflow for any x.  The
// small factor is formed as th * th, th = e^(-|z|), and applied last, one
// factor at a time: th stays a normal number wherever the result is
// representable, so the result rounds once even when it is subnormal (a
// subnormal e^(-2|z|) would carry only a few significant bits).
//
// bf16/fp16 outputs: two values per instruction in packed fp32 (f32x2), with
// the hardware approximations of 2^v and 1/v (ex2.approx, rcp.approx; both
// within ~2^-22 relative) -- th = 2^(-|h|), h = z * log2(e) folded into the
// polynomial's constants.  The error is far below a 16-bit ulp.  fp32 output:
// expf and an IEEE division, each operation rounded to nearest.
//
// The tensor is walked as one flat array: a grid-stride loop of 32-byte (or
// narrower) vector accesses, two vectors in flight per thread, over a grid of
// two vectors per thread; a scalar head when input and output share a
// misalignment; a scalar tail.
#include "dit_device.cuh"
#include "dit_internal.h"

namespace dit {

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kGeluCubic = 0.044715f;
// sqrt(2/pi) * log2(e), and that times 0.044715: h = x * (kH0 + kH1 * x^2)
constexpr float kH0 = 1.1511040990721626f;
constexpr float kH1 = 0.05147161979001175f;

__device__ __forceinline__ float ex2_approx(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// fp32 output: every step rounded to nearest, expf and an IEEE division.
__device__ __forceinline__ float gelu_accurate(float x) {
  const float x2 = __fmul_rn(x, x);
  const float z = __fmul_rn(kSqrt2OverPi, fmaf(__fmul_rn(kGeluCubic, x2), x, x));
  const float th = expf(-fabsf(z));
  const float q = __fdiv_rn(1.0f, fmaf(th, th, 1.0f));
  const float f = z >= 0.0f ? 1.0f : th;
  return __fmul_rn(__fmul_rn(__fmul_rn(x, q), f), f);
}

// 16-bit outputs, one value (heads, tails, 2-byte accesses).
__device__ __forceinline__ float gelu_fast(float x) {
  const float h = __fmul_rn(x, fmaf(kH1, __fmul_rn(x, x), kH0));
  const float th = ex2_approx(-fabsf(h));
  const float q = rcp_approx(fmaf(th, th, 1.0f));
  const float f = h >= 0.0f ? 1.0f : th;
  return __fmul_rn(__fmul_rn(__fmul_rn(x, q), f), f);
}

// 16-bit outputs, a pair of values: the same steps as gelu_fast.
__device__ __forceinline__ F2 gelu_fast2(F2 x) {
  const F2 h = f2_mul(x, f2_fma(f2(kH1, kH1), f2_mul(x, x), f2(kH0, kH0)));
  const float h0 = f2_lo(h), h1 = f2_hi(h);
  const float t0 = ex2_approx(-fabsf(h0)), t1 = ex2_approx(-fabsf(h1));
  const F2 th = f2(t0, t1);
  const F2 d = f2_fma(th, th, f2(1.0f, 1.0f));
  const F2 q = f2(rcp_approx(f2_lo(d)), rcp_approx(f2_hi(d)));
  const F2 f = f2(h0 >= 0.0f ? 1.0f : t0, h1 >= 0.0f ? 1.0f : t1);
  return f2_mul(f2_mul(f2_mul(x, q), f), f);
}

template <class T>
__device__ __forceinline__ float gelu_scalar(float x) {
  if constexpr (sizeof(T) == 4) {
    return gelu_accurate(x);
  } else {
    return gelu_fast(x);
  }
}

// VB bytes of T in, VB bytes out.
template <class T, int VB>
__device__ __forceinline__ Raw<VB> gelu_vec(const Raw<VB>& r) {
  if constexpr (sizeof(T) == 2 && VB >= 4) {
    Raw<VB> o;
#pragma unroll
    for (int i = 0; i < VB / 4; ++i) o.w[i] = Pair<T>::narrow(gelu_fast2(Pair<T>::widen(r.w[i])));
    return o;
  } else {
    using V = Vec<T, VB>;
    float x[V::N], y[V::N];
    V::widen(r, x);
#pragma unroll
    for (int e = 0; e < V::N; ++e) y[e] = gelu_scalar<T>(x[e]);
    return V::narrow(y);
  }
}

struct GeluArgs {
  void* out;
  const void* x;
  int64_t n_head;
  int64_t n_vec;
  int64_t n_tail;
};

template <class T, int VB>
__global__ void __launch_bounds__(256) gelu_flat_kernel(GeluArgs a) {
  using S = Vec<T, (int)sizeof(T)>;
  constexpr int ES = (int)sizeof(T);
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;

  if (gtid < a.n_head + a.n_tail) {
    const int64_t i = gtid < a.n_head ? gtid : a.n_head + a.n_vec * (VB / ES) + (gtid - a.n_head);
    float x[1], y[1];
    S::widen(ld_stream<ES>((const char*)a.x + i * ES), x);
    y[0] = gelu_scalar<T>(x[0]);
    st_stream<ES>((char*)a.out + i * ES, S::narrow(y));
  }
  const char* xb = (const char*)a.x + a.n_head * ES;
  char* ob = (char*)a.out + a.n_head * ES;
  int64_t i = gtid;
  // two vectors in flight: both loads issue before either is computed
  for (; i + nthreads < a.n_vec; i += 2 * nthreads) {
    const Raw<VB> r0 = ld_stream<VB>(xb + i * VB);
    const Raw<VB> r1 = ld_stream<VB>(xb + (i + nthreads) * VB);
    st_stream<VB>(ob + i * VB, gelu_vec<T, VB>(r0));
    st_stream<VB>(ob + (i + nthreads) * VB, gelu_vec<T, VB>(r1));
  }
  if (i < a.n_vec) st_stream<VB>(ob + i * VB, gelu_vec<T, VB>(ld_stream<VB>(xb + i * VB)));
}

cudaError_t launch_gelu(const DeviceInfo& dev, int dtype, void* out, const void* x, int64_t n,
                        cudaStream_t stream) {
  const int es = dtype == 2 ? 4 : 2;
  const uint64_t p0 = (uint64_t)(uintptr_t)x;
  const int vb = widest_access(p0 ^ (uint64_t)(uintptr_t)out);
  const int64_t mis = (int64_t)(p0 & (uint64_t)(vb - 1));
  GeluArgs a;
  a.out = out;
  a.x = x;
  a.n_head = mis ? (vb - mis) / es : 0;
  if (a.n_head > n) a.n_head = n;
  const int64_t per_vec = vb / es;
  a.n_vec = (n - a.n_head) / per_vec;
  a.n_tail = n - a.n_head - a.n_vec * per_vec;
  return dispatch_dtype_width(dtype, vb, [&](auto tt, auto w) -> cudaError_t {
    using T = typename decltype(tt)::type;
    constexpr int VB = decltype(w)::value;
    const int block = 256;
    // two vectors per thread (one pass of the loop): short CTAs handed to the
    // SMs by the hardware, as for the full-gate residual gate (a one-wave
    // grid left SMs idle at the end); the loop covers what a grid of at most
    // 2^30 CTAs does not
    int64_t grid = (a.n_vec + 2 * block - 1) / (2 * block);
    if (grid > (int64_t(1) << 30)) grid = int64_t(1) << 30;
    const int64_t edge = (a.n_head + a.n_tail + block - 1) / block;
    if (grid < edge) grid = edge;
    if (grid < 1) grid = 1;
    gelu_flat_kernel<T, VB><<<(unsigned)grid, block, 0, stream>>>(a);
    return cudaGetLastError();
  });
}

}  // namespace dit
