// k_gelu.cu -- tanh-approximated GELU, elementwise, on GB300.
//
// gelu(x) = 0.5 * x * (1 + tanh(z)),  z = sqrt(2/pi) * (x + 0.044715 * x^3):
// the activation of the LTX-2 feed-forward (prhub summary of sglang PR #34172,
// "implementation breakdown" item 3: LTX2FeedForward's tanh-GELU after
// proj_in).  Evaluated as x * sigmoid(2z) -- the same function, since
// 1 + tanh(z) = 2 / (1 + exp(-2z)) -- with sigmoid(2z) = 1/(1+t) for z >= 0
// and t/(1+t) for z < 0, t = exp(-2|z|) in (0, 1]: no cancellation and no
// overflow for any x.
//
// The tensor is walked as one flat array: a grid-stride loop of 32-byte (or
// narrower) vector accesses, a scalar head when input and output share a
// misalignment, a scalar tail.  16-bit outputs use the fast exp and divide
// intrinsics (relative error well under 1e-4, far below a bf16/fp16 ulp);
// fp32 output uses expf and an IEEE division.
#include "dit_device.cuh"
#include "dit_internal.h"

namespace dit {

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kGeluCubic = 0.044715f;

template <bool ACCURATE>
__device__ __forceinline__ float gelu_tanh(float x) {
  const float x2 = __fmul_rn(x, x);
  const float z = __fmul_rn(kSqrt2OverPi, fmaf(__fmul_rn(kGeluCubic, x2), x, x));
  const float az = fabsf(z);
  float t, q;
  if constexpr (ACCURATE) {
    t = expf(-2.0f * az);
    q = 1.0f / (1.0f + t);
  } else {
    t = __expf(-2.0f * az);
    q = __fdividef(1.0f, 1.0f + t);
  }
  const float s = z >= 0.0f ? q : __fmul_rn(t, q);
  return __fmul_rn(x, s);
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
  using V = Vec<T, VB>;
  using S = Vec<T, (int)sizeof(T)>;
  constexpr int N = V::N;
  constexpr int ES = (int)sizeof(T);
  constexpr bool kAccurate = sizeof(T) == 4;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;

  if (gtid < a.n_head + a.n_tail) {
    const int64_t i = gtid < a.n_head ? gtid : a.n_head + a.n_vec * N + (gtid - a.n_head);
    float x[1], y[1];
    S::widen(ld_stream<ES>((const char*)a.x + i * ES), x);
    y[0] = gelu_tanh<kAccurate>(x[0]);
    st_stream<ES>((char*)a.out + i * ES, S::narrow(y));
  }
  const char* xb = (const char*)a.x + a.n_head * ES;
  char* ob = (char*)a.out + a.n_head * ES;
  for (int64_t i = gtid; i < a.n_vec; i += nthreads) {
    float x[N], y[N];
    V::widen(ld_stream<VB>(xb + i * VB), x);
#pragma unroll
    for (int e = 0; e < N; ++e) y[e] = gelu_tanh<kAccurate>(x[e]);
    st_stream<VB>(ob + i * VB, V::narrow(y));
  }
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
    const void* fn = (const void*)gelu_flat_kernel<T, VB>;
    const int block = 256;
    int64_t grid = (a.n_vec + block - 1) / block;
    const int64_t wave = (int64_t)dev.sm_count * resident_ctas(dev, fn, block);
    if (grid > wave) grid = wave;
    const int64_t edge = (a.n_head + a.n_tail + block - 1) / block;
    if (grid < edge) grid = edge;
    if (grid < 1) grid = 1;
    gelu_flat_kernel<T, VB><<<(unsigned)grid, block, 0, stream>>>(a);
    return cudaGetLastError();
  });
}

}  // namespace dit
