// dit_pipe.cuh -- shared-memory-staged row kernels (16-byte aligned rows).
//
// Each thread streams the 16-byte granules it owns -- granules t + k * T of
// every row, k < VPT, for T threads -- from HBM into its own slots of an
// S-stage shared-memory ring with cp.async, RC rows per stage.  Stages are
// issued S-1 groups ahead of the one being computed, so up to
// (S-1) * RC * VPT * 16 bytes per thread per streamed operand are in flight
// while registers hold only the group being computed.  A thread only ever
// reads the slots it filled itself, so cp.async.wait_group (a hardware wait:
// no spin loop) is the only synchronisation the ring needs; the one
// __syncthreads per group belongs to the row reduction.
//
// The [B, 1, D] operands are loaded once per CTA and kept in registers in
// fp32, with 1 + scale already formed (one fp32 rounding, as in the
// modulation's definition).  The modulation takes two passes over the staged
// row: sum of squares, then -- after the reduction -- normalise, modulate and
// store.  The fused op computes the residual in pass one, stores it to HBM,
// writes it back over its own hidden slot, and pass two reads it from there.
#pragma once

#include "dit_device.cuh"
#include "dit_internal.h"

namespace dit {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ Raw<16> lds16(const Raw<16>* p) {
  Raw<16> r;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
               : "r"(smem_addr(p)));
  return r;
}
__device__ __forceinline__ void sts16(Raw<16>* p, const Raw<16>& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_addr(p)), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
               : "memory");
}

// Streamed operands of each operation (in ring slot order).
template <int OP, bool GFULL, bool MFULL>
__host__ __device__ constexpr int streamed_operands() {
  return OP == OP_MOD ? (MFULL ? 3 : 1) : OP == OP_RGA ? 2 : (2 + (GFULL ? 1 : 0) + (MFULL ? 2 : 0));
}

template <int OP, class T, int VPT, int S, int RC, bool GFULL, bool MFULL>
__global__ void __launch_bounds__(512) pipe_kernel(RowArgs a) {
  using V = Vec<T, 16>;
  constexpr int NE = V::N;  // elements per granule
  constexpr int NS = streamed_operands<OP, GFULL, MFULL>();
  constexpr bool kReduce = OP != OP_RGA;
  constexpr bool kGate = OP != OP_MOD;
  // ring slot index of each operand
  constexpr int kX = 0;                                 // hidden / x
  constexpr int kU = 1;                                 // update
  constexpr int kG = 2;                                 // full gate
  constexpr int kSc = (OP == OP_MOD) ? 1 : (GFULL ? 3 : 2);  // full scale
  constexpr int kSh = kSc + 1;                          // full shift

  extern __shared__ Raw<16> ring[];  // [S][RC][NS][VPT][T]
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;

  const int64_t b = blockIdx.x / a.chunks_per_batch;
  const int64_t chunk = blockIdx.x - b * a.chunks_per_batch;
  const int64_t r_begin = b * a.L + chunk * a.rows_per_chunk;
  const int64_t r_stop = (b + 1) * a.L;
  const int64_t r_end = r_begin + a.rows_per_chunk < r_stop ? r_begin + a.rows_per_chunk : r_stop;
  if (r_begin >= r_end) return;  // uniform over the CTA
  const int64_t pitch = a.D * (int64_t)sizeof(T);
  const int64_t col0 = (int64_t)blockIdx.y * nthr * VPT;  // column slices (residual gate)

  int64_t coff[VPT];
  bool cval[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int64_t cg = col0 + tid + (int64_t)k * nthr;
    cval[k] = cg < a.nvec;
    coff[k] = cg * 16;
  }

  // [B, 1, D] operands in fp32 registers
  float gv[VPT][NE], onev[VPT][NE], shv[VPT][NE];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    if (!cval[k]) continue;
    if constexpr (kGate && !GFULL) V::widen(ld_bcast<16>((const char*)a.g + b * pitch + coff[k]), gv[k]);
    if constexpr (kReduce && !MFULL) {
      V::widen(ld_bcast<16>((const char*)a.sc + b * pitch + coff[k]), onev[k]);
#pragma unroll
      for (int e = 0; e < NE; ++e) onev[k][e] = __fadd_rn(1.0f, onev[k][e]);
      V::widen(ld_bcast<16>((const char*)a.sh + b * pitch + coff[k]), shv[k]);
    }
  }

  const void* src[5] = {a.x, a.u, a.g, a.sc, a.sh};
  const char* sptr[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    int which = i;
    if (OP == OP_MOD && i >= 1) which = 2 + i;       // x, scale, shift
    if (OP == OP_FUSED && !GFULL && i >= 2) which = i + 1;  // h, u, scale, shift
    sptr[i] = (const char*)src[which];
  }
  auto slot = [&](int stage, int j, int op, int k) -> Raw<16>* {
    return ring + (((stage * RC + j) * NS + op) * VPT + k) * nthr + tid;
  };

  const int64_t ngroups = (r_end - r_begin + RC - 1) / RC;
  auto issue = [&](int64_t grp) {
    if (grp < ngroups) {
      const int stage = (int)(grp % S);
#pragma unroll
      for (int j = 0; j < RC; ++j) {
        const int64_t row = r_begin + grp * RC + j;
        if (row >= r_end) continue;
        const int64_t rowoff = row * pitch;
#pragma unroll
        for (int op = 0; op < NS; ++op)
#pragma unroll
          for (int k = 0; k < VPT; ++k)
            if (cval[k]) cp_async16(smem_addr(slot(stage, j, op, k)), sptr[op] + rowoff + coff[k]);
      }
    }
    cp_async_commit();  // possibly empty: keeps the group count uniform
  };

#pragma unroll
  for (int s = 0; s < S - 1; ++s) issue(s);

  __shared__ float part[2][RC][16];  // per-warp partial sums (<= 16 warps)
  int buf = 0;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = nthr >> 5;

  for (int64_t grp = 0; grp < ngroups; ++grp) {
    cp_async_wait<S - 2>();  // group grp has landed (for this thread's slots)
    const int stage = (int)(grp % S);
    // refill the stage consumed in the previous iteration
    issue(grp + S - 1);

    float ss[RC];
#pragma unroll
    for (int j = 0; j < RC; ++j) {
      ss[j] = 0.0f;
      const int64_t row = r_begin + grp * RC + j;
      if (row >= r_end) continue;
      const int64_t rowoff = row * pitch;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!cval[k]) continue;
        float x[NE];
        if constexpr (kGate) {
          float h[NE], u[NE], gf[NE];
          V::widen(lds16(slot(stage, j, kX, k)), h);
          V::widen(lds16(slot(stage, j, kU, k)), u);
          if constexpr (GFULL) V::widen(lds16(slot(stage, j, kG, k)), gf);
#pragma unroll
          for (int e = 0; e < NE; ++e) x[e] = residual_gate(h[e], u[e], GFULL ? gf[e] : gv[k][e]);
          const Raw<16> r = V::narrow(x);
          st_stream<16>((char*)a.out + rowoff + coff[k], r);
          if constexpr (kReduce) {
            sts16(slot(stage, j, kX, k), r);  // the stored residual, for pass two
            V::widen(r, x);
          }
        } else {
          V::widen(lds16(slot(stage, j, kX, k)), x);
        }
        if constexpr (kReduce) {
#pragma unroll
          for (int e = 0; e < NE; ++e) ss[j] = fmaf(x[e], x[e], ss[j]);
        }
      }
    }
    if constexpr (kReduce) {
#pragma unroll
      for (int j = 0; j < RC; ++j) {
        const float w = warp_sum(ss[j]);
        if (lane == 0) part[buf][j][warp] = w;
      }
      __syncthreads();
      float rinv[RC];
#pragma unroll
      for (int j = 0; j < RC; ++j) {
        float tot = 0.0f;
        for (int w = 0; w < nwarps; ++w) tot += part[buf][j][w];
        rinv[j] = rms_inverse(tot, a.D, a.eps);
      }
      buf ^= 1;
      void* mout = OP == OP_FUSED ? a.out2 : a.out;
#pragma unroll
      for (int j = 0; j < RC; ++j) {
        const int64_t row = r_begin + grp * RC + j;
        if (row >= r_end) continue;
        const int64_t rowoff = row * pitch;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          if (!cval[k]) continue;
          float x[NE], y[NE];
          V::widen(lds16(slot(stage, j, kX, k)), x);
          if constexpr (MFULL) {
            float s[NE], h[NE];
            V::widen(lds16(slot(stage, j, kSc, k)), s);
            V::widen(lds16(slot(stage, j, kSh, k)), h);
#pragma unroll
            for (int e = 0; e < NE; ++e) y[e] = modulate(x[e], rinv[j], s[e], h[e]);
          } else {
#pragma unroll
            for (int e = 0; e < NE; ++e)
              y[e] = __fadd_rn(__fmul_rn(__fmul_rn(x[e], rinv[j]), onev[k][e]), shv[k][e]);
          }
          st_stream<16>((char*)mout + rowoff + coff[k], V::narrow(y));
        }
      }
    }
  }
  cp_async_wait<0>();  // no copy may outlive the CTA's shared memory
}

// Stages and rows per stage of each operation (tuning builds may override).
#ifndef DIT_PIPE_S_RGA
#define DIT_PIPE_S_RGA 4
#endif
#ifndef DIT_PIPE_RC_RGA
#define DIT_PIPE_RC_RGA 1
#endif
#ifndef DIT_PIPE_S_MOD
#define DIT_PIPE_S_MOD 4
#endif
#ifndef DIT_PIPE_RC_MOD
#define DIT_PIPE_RC_MOD 2
#endif
#ifndef DIT_PIPE_S_FUSED
#define DIT_PIPE_S_FUSED 3
#endif
#ifndef DIT_PIPE_RC_FUSED
#define DIT_PIPE_RC_FUSED 2
#endif
constexpr int kPipeVPT = 2;           // 16-byte granules per thread per row
constexpr int kPipeBlockMax = 512;    // threads: rows up to 16 KB
constexpr int kStaticSmemReserve = 1024;  // bytes kept for the static arrays

template <int OP>
__host__ __device__ constexpr int pipe_stages() {
  return OP == OP_RGA ? DIT_PIPE_S_RGA : OP == OP_MOD ? DIT_PIPE_S_MOD : DIT_PIPE_S_FUSED;
}
template <int OP>
__host__ __device__ constexpr int pipe_rows() {
  return OP == OP_RGA ? DIT_PIPE_RC_RGA : OP == OP_MOD ? DIT_PIPE_RC_MOD : DIT_PIPE_RC_FUSED;
}

// Launch the staged kernel with S stages; returns cudaErrorNotSupported when
// the row is too long for it (the caller then uses the two-pass kernel).
template <int OP, class T, int S, bool GFULL, bool MFULL>
cudaError_t launch_pipe_s(const DeviceInfo& dev, RowArgs a, int64_t B, int block,
                          unsigned slices, size_t smem, cudaStream_t stream) {
  constexpr int RC = pipe_rows<OP>();
  auto kern = pipe_kernel<OP, T, kPipeVPT, S, RC, GFULL, MFULL>;
  // allow the ring's dynamic shared memory: raised per device as needed
  static size_t configured[64];
  const bool cached = dev.device >= 0 && dev.device < 64;
  // (the default limit, 48 KB, covers static and dynamic shared memory together)
  if (smem + kStaticSmemReserve > 48 * 1024 && (!cached || configured[dev.device] < smem)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();  // do not leave it for the next call to report
      return e;
    }
    if (cached) configured[dev.device] = smem;
  }
  RowPlan plan;
  if (!plan_rows(dev, (const void*)kern, block, B, a.L, slices, &plan, smem))
    return cudaErrorInvalidConfiguration;
  a.rows_per_chunk = plan.rows_per_chunk;
  a.chunks_per_batch = plan.chunks_per_batch;
  kern<<<plan.grid, plan.block, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int OP, bool GFULL, bool MFULL>
cudaError_t launch_pipe(const DeviceInfo& dev, int dtype, RowArgs a, int64_t B,
                        cudaStream_t stream) {
  constexpr int NS = streamed_operands<OP, GFULL, MFULL>();
  constexpr int RC = pipe_rows<OP>();
  const int64_t row_bytes = a.D * (dtype == 2 ? 4 : 2);
  a.nvec = row_bytes / 16;
  const int64_t threads_needed = (a.nvec + kPipeVPT - 1) / kPipeVPT;
  int block;
  unsigned slices = 1;
  if (OP == OP_RGA) {
    block = (int)((threads_needed < 256 ? threads_needed : 256) + 31) / 32 * 32;
    const int64_t s = (a.nvec + (int64_t)block * kPipeVPT - 1) / ((int64_t)block * kPipeVPT);
    if (s > 65535) return cudaErrorInvalidConfiguration;
    slices = (unsigned)s;
  } else {
    if (threads_needed > kPipeBlockMax) return cudaErrorNotSupported;
    block = (int)((threads_needed + 31) / 32 * 32);
  }
  const size_t per_stage = (size_t)RC * NS * kPipeVPT * block * 16;
  const size_t limit = (size_t)(dev.smem_optin - kStaticSmemReserve);
  int S = pipe_stages<OP>();
  while (S > 2 && per_stage * S > limit) S = S > 3 ? 3 : 2;
  if (per_stage * S > limit) return cudaErrorNotSupported;
  // instantiated stage counts: 2, 3 and the operation's default
  return dispatch_dtype_width(dtype, 16, [&](auto tt, auto) -> cudaError_t {
    using T = typename decltype(tt)::type;
    constexpr int SD = pipe_stages<OP>();
    if (S == 2) return launch_pipe_s<OP, T, 2, GFULL, MFULL>(dev, a, B, block, slices, 2 * per_stage, stream);
    if constexpr (SD > 3)
      if (S == SD) return launch_pipe_s<OP, T, SD, GFULL, MFULL>(dev, a, B, block, slices, SD * per_stage, stream);
    return launch_pipe_s<OP, T, 3, GFULL, MFULL>(dev, a, B, block, slices, 3 * per_stage, stream);
  });
}

}  // namespace dit
