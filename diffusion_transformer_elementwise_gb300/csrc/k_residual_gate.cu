// k_residual_gate.cu -- out = hidden + update * gate on GB300.
//
// Operation: sglang PR #29361 "Add diffusion residual-gate CUDA fast path for
// LTX2", section Motivation (hidden + update * gate over contiguous
// [B, L, D] tensors, with a full gate or a [B, 1, D] gate).
//
// Full gate: the four tensors are walked as one flat array.  Every element
// has the same index in all of them, so the kernel is a grid-stride loop of
// 32-byte (or narrower) vector loads with no index arithmetic beyond the
// stride, over a grid of one vector per thread.  When the pointers share their misalignment, a scalar head brings
// the body onto the vector boundary; a scalar tail finishes it.
//
// Row-broadcast gate: the row-tiled kernel of dit_rows.cuh (OP_RGA), which
// keeps each CTA's slice of the gate in registers across its rows.  The page's
// B200 kernel reused the gate across 4 rows and removed a per-element modulo
// (section "Speed Tests and Profiling", B200 Nsight Compute table); here a
// CTA reuses it across its whole run of rows and no index is ever divided.
#include "dit_rows.cuh"

namespace dit {

template <class T, int VB, int U>
__global__ void __launch_bounds__(256) rga_flat_kernel(FlatArgs a) {
  using V = Vec<T, VB>;
  using S = Vec<T, (int)sizeof(T)>;
  constexpr int N = V::N;
  constexpr int ES = (int)sizeof(T);
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;

  // scalar head and tail elements, one per thread
  if (gtid < a.n_head + a.n_tail) {
    const int64_t i = gtid < a.n_head ? gtid : a.n_head + a.n_vec * N + (gtid - a.n_head);
    float h[1], u[1], g[1], y[1];
    S::widen(ld_stream<ES>((const char*)a.h + i * ES), h);
    S::widen(ld_stream<ES>((const char*)a.u + i * ES), u);
    S::widen(ld_stream<ES>((const char*)a.g + i * ES), g);
    y[0] = residual_gate(h[0], u[0], g[0]);
    st_stream<ES>((char*)a.out + i * ES, S::narrow(y));
  }

  const int64_t body = a.n_head * ES;
  const char* hb = (const char*)a.h + body;
  const char* ub = (const char*)a.u + body;
  const char* gb = (const char*)a.g + body;
  char* ob = (char*)a.out + body;
  for (int64_t base = gtid; base < a.n_vec; base += nthreads * U) {
    Raw<VB> hv[U], uv[U], gv[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t i = base + k * nthreads;
      if (i < a.n_vec) {
        hv[k] = ld_stream<VB>(hb + i * VB);
        uv[k] = ld_stream<VB>(ub + i * VB);
        gv[k] = ld_stream<VB>(gb + i * VB);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t i = base + k * nthreads;
      if (i < a.n_vec) {
        float h[N], u[N], g[N], y[N];
        V::widen(hv[k], h);
        V::widen(uv[k], u);
        V::widen(gv[k], g);
#pragma unroll
        for (int e = 0; e < N; ++e) y[e] = residual_gate(h[e], u[e], g[e]);
        st_stream<VB>(ob + i * VB, V::narrow(y));
      }
    }
  }
}

constexpr int kFlatUnroll = 1;
constexpr int kFlatBlock = 256;

cudaError_t launch_rga_full(const DeviceInfo& dev, int dtype, void* out, const void* h,
                            const void* u, const void* g, int64_t n, cudaStream_t stream) {
  const int es = dtype == 2 ? 4 : 2;
  const uint64_t p0 = (uint64_t)(uintptr_t)h;
  // pointers that share their offset modulo the access width can all be
  // brought onto that boundary by the same scalar head
  const uint64_t diff = (p0 ^ (uint64_t)(uintptr_t)out) | (p0 ^ (uint64_t)(uintptr_t)u) |
                        (p0 ^ (uint64_t)(uintptr_t)g);
  const int vb = widest_access(diff);
  const int64_t mis = (int64_t)(p0 & (uint64_t)(vb - 1));
  FlatArgs a;
  a.out = out;
  a.h = h;
  a.u = u;
  a.g = g;
  a.n_head = mis ? (vb - mis) / es : 0;
  if (a.n_head > n) a.n_head = n;
  const int64_t per_vec = vb / es;
  a.n_vec = (n - a.n_head) / per_vec;
  a.n_tail = n - a.n_head - a.n_vec * per_vec;
  return dispatch_dtype_width(dtype, vb, [&](auto tt, auto w) -> cudaError_t {
    using T = typename decltype(tt)::type;
    constexpr int VB = decltype(w)::value;
    // one vector per thread: short CTAs handed to the SMs by the hardware as
    // earlier ones finish.  A one-wave grid striding over the tensors left
    // SMs idle at the end (ncu: 219k to 303k active cycles per SM) --
    // [1,32640,4096] bf16 back to back 154.9 -> 147.5 us.  The grid-stride
    // loop covers what a grid of at most 2^30 CTAs does not.
    const int64_t per_cta = (int64_t)kFlatBlock * kFlatUnroll;
    int64_t grid = (a.n_vec + per_cta - 1) / per_cta;
    if (grid > (int64_t(1) << 30)) grid = int64_t(1) << 30;
    const int64_t edge = (a.n_head + a.n_tail + kFlatBlock - 1) / kFlatBlock;
    if (grid < edge) grid = edge;
    if (grid < 1) grid = 1;
    rga_flat_kernel<T, VB, kFlatUnroll><<<(unsigned)grid, kFlatBlock, 0, stream>>>(a);
    return cudaGetLastError();
  });
}

cudaError_t launch_rga_bcast(const DeviceInfo& dev, int dtype, int vb, const RowArgs& a,
                             int64_t B, cudaStream_t stream) {
  return launch_row_op<OP_RGA, false, false>(dev, dtype, vb, a, B, stream);
}

cudaError_t launch_rga_grouped(const DeviceInfo& dev, int dtype, const RowArgs* a,
                               const int64_t* B, int count, cudaStream_t stream) {
  return launch_pipe_grouped<OP_RGA, false, false, false>(dev, dtype, a, B, count, stream);
}

}  // namespace dit
