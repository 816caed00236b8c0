// dit_warprow.cuh -- modulation with one warp per row (16-byte aligned rows,
// [B, 1, D] scale and shift).
//
// Each warp owns whole rows: lane l handles the 16-byte granules l, l+32, ...
// of the row, so the row's sum of squares needs only the warp's shuffles --
// no shared-memory partials and no CTA barrier per row.  Each warp streams its
// rows from HBM into its own shared-memory ring with cp.async (S stages, one
// row per stage; hardware waits, no spin loop).
//
// 1 + scale (formed once, one fp32 rounding) and shift are kept in shared
// memory as fp32 for the whole CTA, laid out so that the 32 lanes of a warp
// read 32 consecutive 16-byte words (conflict-free).  The CTA takes groups of
// W consecutive rows of one batch (one per warp), groups c, c+G, c+2G, ...;
// all warps step through the same groups, so the vectors are reloaded -- the
// only CTA barriers -- exactly when the group's batch changes.
#pragma once

#include "dit_pipe.cuh"

namespace dit {

template <class T, int S>
__global__ void __maxnreg__(96) warp_mod_kernel(RowArgs a) {  // <= 16 warps x 96 registers
  using G = Granule<T>;
  constexpr int P = G::P;  // fp32 pairs per granule
  constexpr int Q = P / 2;  // float4 per granule
  extern __shared__ __align__(16) float4 wsm[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int W = blockDim.x >> 5;
  const int64_t nvec = a.nvec;              // granules per row
  const int ng_full = (int)(nvec >> 5);     // granules every lane has
  const int tail = (int)(nvec & 31);        // lanes with one more
  const int ng = ng_full + (tail ? 1 : 0);

  // shared memory: (1 + scale) and shift [ng][Q][32] float4 each, then the
  // rings [W][S][ng][32] of 16-byte granules
  float4* const onev = wsm;
  float4* const shv = wsm + ng * Q * 32;
  const uint32_t stage_bytes = (uint32_t)ng * 512;
  const uint32_t ring = smem_addr(wsm + 2 * ng * Q * 32) + (uint32_t)warp * S * stage_bytes +
                        (uint32_t)lane * 16;
  const uint32_t ring_end = ring + S * stage_bytes;
  const int64_t pitch = a.D * (int64_t)sizeof(T);
  const char* const xg = (const char*)a.x + (int64_t)lane * 16;
  char* const og = (char*)a.out + (int64_t)lane * 16;
  const bool has_tail = lane < tail;

  const int64_t nbatch = a.ngroups / a.gpb;
  auto advance = [&](int64_t& bb, int64_t& gg) {
    bb += a.step_b;
    gg += a.step_g;
    if (gg >= a.gpb) {
      gg -= a.gpb;
      ++bb;
    }
  };

  int64_t ib = (int64_t)blockIdx.x / a.gpb, ig = (int64_t)blockIdx.x - ib * a.gpb;
  uint32_t istage = ring;
  auto issue = [&]() {
    if (ib < nbatch) {
      const int64_t row = ib * a.L + ig * W + warp;
      if (row < (ib + 1) * a.L) {
        const char* src = xg + row * pitch;
        for (int k = 0; k < ng_full; ++k) cp_async16(istage + k * 512, src + k * 512);
        if (has_tail) cp_async16(istage + ng_full * 512, src + ng_full * 512);
      }
    }
    cp_async_commit();  // possibly empty: keeps the group count uniform
    advance(ib, ig);
    istage = istage + stage_bytes == ring_end ? ring : istage + stage_bytes;
  };

  // vectors of batch bb, by all threads of the CTA
  auto load_vectors = [&](int64_t bb) {
    __syncthreads();  // every warp is done with the previous batch's vectors
    for (int64_t gi = threadIdx.x; gi < nvec; gi += blockDim.x) {
      F2 s[P], h[P];
      G::widen(ld_bcast<16>((const char*)a.sc + bb * pitch + gi * 16), s);
      G::widen(ld_bcast<16>((const char*)a.sh + bb * pitch + gi * 16), h);
      const int k = (int)(gi >> 5), ln = (int)(gi & 31);
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const F2 o0 = f2_add(f2(1.0f, 1.0f), s[2 * q]);
        const F2 o1 = f2_add(f2(1.0f, 1.0f), s[2 * q + 1]);
        onev[(k * Q + q) * 32 + ln] = make_float4(f2_lo(o0), f2_hi(o0), f2_lo(o1), f2_hi(o1));
        shv[(k * Q + q) * 32 + ln] =
            make_float4(f2_lo(h[2 * q]), f2_hi(h[2 * q]), f2_lo(h[2 * q + 1]), f2_hi(h[2 * q + 1]));
      }
    }
    __syncthreads();
  };

  // one granule: pass two (normalise, modulate, narrow, store)
  auto emit = [&](uint32_t sl, int k, F2 r2, char* dst) {
    F2 x[P], y[P];
    G::widen(lds16(sl), x);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float4 o = onev[(k * Q + q) * 32 + lane];
      const float4 h = shv[(k * Q + q) * 32 + lane];
      y[2 * q] = modulate2(f2_mul(x[2 * q], r2), f2(o.x, o.y), f2(h.x, h.y));
      y[2 * q + 1] = modulate2(f2_mul(x[2 * q + 1], r2), f2(o.z, o.w), f2(h.z, h.w));
    }
    st_stream<16>(dst, G::narrow(y));
  };

#pragma unroll
  for (int s = 0; s < S - 1; ++s) issue();

  int64_t cb = (int64_t)blockIdx.x / a.gpb, cg = (int64_t)blockIdx.x - cb * a.gpb;
  int64_t vec_b = -1;
  uint32_t stage = ring;
  while (cb < nbatch) {
    cp_async_wait<S - 2>();  // this lane's copies of this row have landed
    issue();
    if (cb != vec_b) {  // uniform over the CTA
      load_vectors(cb);
      vec_b = cb;
    }
    const int64_t row = cb * a.L + cg * W + warp;
    if (row < (cb + 1) * a.L) {  // uniform over the warp
      // pass one: sum of squares
      F2 acc[P];
#pragma unroll
      for (int i = 0; i < P; ++i) acc[i] = f2(0.0f, 0.0f);
#pragma unroll 4
      for (int k = 0; k < ng_full; ++k) {
        F2 x[P];
        G::widen(lds16(stage + k * 512), x);
#pragma unroll
        for (int i = 0; i < P; ++i) acc[i] = f2_fma(x[i], x[i], acc[i]);
      }
      if (has_tail) {
        F2 x[P];
        G::widen(lds16(stage + ng_full * 512), x);
#pragma unroll
        for (int i = 0; i < P; ++i) acc[i] = f2_fma(x[i], x[i], acc[i]);
      }
#pragma unroll
      for (int i = 1; i < P; ++i) acc[0] = f2_add(acc[0], acc[i]);
      const float tot = warp_sum(f2_lo(acc[0]) + f2_hi(acc[0]));
      const float r = rms_inverse(tot, a.d_f, a.inv_d, a.eps);
      const F2 r2 = f2(r, r);
      // pass two
      char* const dst = og + row * pitch;
#pragma unroll 4
      for (int k = 0; k < ng_full; ++k) emit(stage + k * 512, k, r2, dst + k * 512);
      if (has_tail) emit(stage + ng_full * 512, ng_full, r2, dst + ng_full * 512);
    }
    stage = stage + stage_bytes == ring_end ? ring : stage + stage_bytes;
    advance(cb, cg);
  }
  cp_async_wait<0>();  // no copy may outlive the CTA's shared memory
}

#ifndef DIT_WARP_STAGES
#define DIT_WARP_STAGES 2
#endif

// Launch the one-warp-per-row modulation; cudaErrorNotSupported when the row
// does not fit (the caller then uses the CTA-per-row kernel).
inline size_t warp_mod_smem(int64_t nvec, int warps, int stages, int q) {
  const int64_t ng = (nvec + 31) / 32;
  return (size_t)(2 * ng * q * 32 * 16) + (size_t)warps * stages * ng * 512;
}

template <class T>
cudaError_t launch_warp_mod(const DeviceInfo& dev, RowArgs a, int64_t B, cudaStream_t stream) {
  constexpr int S = DIT_WARP_STAGES;
  constexpr int Q = Granule<T>::P / 2;
  const int64_t row_bytes = a.D * (int64_t)sizeof(T);
  a.nvec = row_bytes / 16;
  const size_t limit = (size_t)(dev.smem_optin - kStaticSmemReserve);
  // as many warps (rows in flight) as one CTA's shared memory holds, up to 16
  int W = 16;
  while (W > 0 && warp_mod_smem(a.nvec, W, S, Q) > limit) --W;
  if (W < 4) return cudaErrorNotSupported;
  const size_t smem = warp_mod_smem(a.nvec, W, S, Q);
  auto kern = warp_mod_kernel<T, S>;
  static size_t configured[64];
  const bool cached = dev.device >= 0 && dev.device < 64;
  if (smem + kStaticSmemReserve > 48 * 1024 && (!cached || configured[dev.device] < smem)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return e;
    }
    if (cached) configured[dev.device] = smem;
  }
  const int block = W * 32;
  a.gpb = (a.L + W - 1) / W;
  a.ngroups = B * a.gpb;
  int64_t Gn = (int64_t)dev.sm_count * resident_ctas(dev, (const void*)kern, block, smem);
  if (Gn > a.ngroups) Gn = a.ngroups;
  if (Gn < 1) Gn = 1;
  if (Gn > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  a.step_b = Gn / a.gpb;
  a.step_g = Gn - a.step_b * a.gpb;
  kern<<<(unsigned)Gn, block, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dit
