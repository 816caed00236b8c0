// dit_rows.cuh -- row-tiled kernels for the residual gate with a [B, 1, D]
// gate, the adaLN RMSNorm-modulation and the fused op.
//
// Tiling.  A CTA takes groups of R consecutive rows of one batch, groups
// c, c + G, c + 2G, ... of a one-wave grid (so the CTAs stream one moving
// window of the tensors), keeps each [B, 1, D] vector in registers across its
// rows (reloaded only when the batch changes; no per-element index
// arithmetic), and owns a column slice of
// blockDim.x * 32 bytes (16 for narrow accesses).  Thread t owns the 32/VB
// (16/VB) vectors of VB bytes at
// vector indices col0 + t + k * blockDim.x: each warp-wide access is
// contiguous.  R rows are in flight per thread (R * 32 bytes per streamed
// operand), which with one wave of resident CTAs keeps enough bytes in
// flight per SM to cover HBM latency.
//
// Reduction (modulation, fused).  The CTA spans the whole row (one column
// slice).  Each thread sums x^2 over its elements in fp32, the warp reduces
// with shuffles, the warps' partials go through shared memory (double
// buffered, so one __syncthreads per R rows), and every thread adds the
// partials in the same order, so all threads hold the same sum.
//
// Long rows (more than kRowBlockMax threads * 32 (16) bytes) use long_row_kernel: one CTA
// per row at a time, a first pass that accumulates the sum of squares (and,
// for the fused op, writes the residual), and a second pass that re-reads the
// row -- for the fused op its own residual writes -- and writes the output.
#pragma once

#include "dit_device.cuh"
#include "dit_internal.h"
#include "dit_pipe.cuh"
#include "dit_wrow.cuh"

namespace dit {

// Bytes of a row per thread per operand: 32 for 16/32-byte accesses, 16 for
// the narrow accesses of unaligned rows (which would otherwise need too many
// registers for their per-vector offsets).
template <int VB>
__host__ __device__ constexpr int thread_bytes() {
  return VB >= 16 ? 32 : 16;
}

constexpr int kRowBlockMax = 512;  // threads; rows up to 16 KB stay in registers

// Register budget of the row kernel: by default the launch bound alone (up to
// 128 registers at 512 threads); DIT_ROW_MAXNREG caps it for tuning builds.
// With 2-byte accesses the default holds it to 64 registers (two CTAs of up
// to 512 threads per SM): the bf16 modulation of 2-byte aligned rows took 86
// registers unbounded, one 416-thread CTA per SM, and ran at two thirds of
// the fp16 kernel's speed (bounded: [1,4097,3077] 53.9 -> 39.6 us).  Wider
// accesses were slower with the bound and keep the plain one.
template <int VB>
constexpr int row_min_blocks() { return VB == 2 ? 2 : 1; }
#ifdef DIT_ROW_MAXNREG
#define DIT_ROW_BOUNDS(VB) __maxnreg__(DIT_ROW_MAXNREG)
#else
#define DIT_ROW_BOUNDS(VB) __launch_bounds__(kRowBlockMax, row_min_blocks<VB>())
#endif

template <int OP, class T, int VB, int R, bool GFULL, bool MFULL, bool EX>
__global__ void DIT_ROW_BOUNDS(VB) row_kernel(RowArgs a) {
  using V = Vec<T, VB>;
  constexpr int N = V::N;
  constexpr int VPT = thread_bytes<VB>() / VB;
  constexpr bool kReduce = OP != OP_RGA;
  constexpr bool kHasGate = OP != OP_MOD;

  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  if ((int64_t)blockIdx.x >= a.ngroups) return;  // uniform over the CTA

  const int64_t pitch = a.D * (int64_t)sizeof(T);
  const int64_t col0 = (int64_t)blockIdx.y * nthr * VPT;
  int64_t coff[VPT];
  bool cval[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int64_t cv = col0 + tid + (int64_t)k * nthr;
    cval[k] = cv < a.nvec;
    coff[k] = cv * VB;
  }

  // [B, 1, D] operands of the current batch, in registers
  Raw<VB> gb[VPT], scb[VPT], shb[VPT];
  auto load_vectors = [&](int64_t b) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (!cval[k]) continue;
      if constexpr (kHasGate && !GFULL) gb[k] = ld_bcast<VB>((const char*)a.g + b * a.vstride + coff[k]);
      if constexpr (kReduce && !MFULL) {
        scb[k] = ld_bcast<VB>((const char*)a.sc + b * a.vstride + coff[k]);
        shb[k] = ld_bcast<VB>((const char*)a.sh + b * a.vstride + coff[k]);
      }
    }
  };

  __shared__ SumPair part[2][R][16];       // per-warp row pairs (<= 16 warps)
  __shared__ uint64_t exact_scratch[16];   // the exact path's warp totals
  __shared__ float partf[2][R][16];        // the fast statistic's warp sums
  __shared__ float part_scaled[16];         // and its rescaled sums (rare)
  for (int i = tid; i < 2 * R * 16; i += nthr)
    if ((i & 15) >= (nthr >> 5)) (&part[0][0][0])[i] = SumPair{0.0f, 0.0f};
  const int nwarps = nthr >> 5;
  // the statistic: four scalar (hi, lo) accumulators per thread and row,
  // element e of the thread's row part into accumulator e % 4
  using Acc = Sq32<4>;
  constexpr int kTerms = (VPT * N + 3) / 4;
  [[maybe_unused]] const float coef = Acc::coef(kTerms);
  constexpr int kLevels = 2 + 5 + 4;  // thread, warp, 16 warps
  int buf = 0;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  // grid-stride over groups of R rows (never straddling a batch): CTA c takes
  // groups c, c + G, c + 2G, ...
  const int64_t nbatch = a.ngroups / a.gpb;
  int64_t cb = (int64_t)blockIdx.x / a.gpb, cg = (int64_t)blockIdx.x - cb * a.gpb;
  int64_t vec_b = -1;
  for (; cb < nbatch;) {
    if (cb != vec_b) {
      load_vectors(cb);
      vec_b = cb;
    }
    const int64_t r0 = cb * a.L + cg * R;
    const int64_t r_end = r0 + R < (cb + 1) * a.L ? r0 + R : (cb + 1) * a.L;
    cb += a.step_b;
    cg += a.step_g;
    if (cg >= a.gpb) {
      cg -= a.gpb;
      ++cb;
    }
    Raw<VB> xv[R][VPT], uv[R][VPT], gv[R][VPT], scv[R][VPT], shv[R][VPT];
    bool rval[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      rval[j] = r0 + j < r_end;
      const int64_t rowoff = (r0 + j) * pitch;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!(rval[j] && cval[k])) continue;
        const int64_t off = rowoff + coff[k];
        xv[j][k] = ld_stream<VB>((const char*)a.x + off);
        if constexpr (kHasGate) uv[j][k] = ld_stream<VB>((const char*)a.u + off);
        if constexpr (kHasGate && GFULL) gv[j][k] = ld_stream<VB>((const char*)a.g + off);
        if constexpr (kReduce && MFULL) {
          scv[j][k] = ld_stream<VB>((const char*)a.sc + off);
          shv[j][k] = ld_stream<VB>((const char*)a.sh + off);
        }
      }
    }

    SumPair ss[R];
    [[maybe_unused]] float ssf[R];  // the fast statistic: one FMA chain per row
#pragma unroll
    for (int j = 0; j < R; ++j) {
      Acc acc;
      acc.zero();
      ssf[j] = 0.0f;
      const int64_t rowoff = (r0 + j) * pitch;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!(rval[j] && cval[k])) continue;
        float f[N];
        if constexpr (kHasGate) {
          float h[N], u[N], g[N];
          V::widen(xv[j][k], h);
          V::widen(uv[j][k], u);
          V::widen(GFULL ? gv[j][k] : gb[k], g);
#pragma unroll
          for (int e = 0; e < N; ++e) f[e] = residual_gate(h[e], u[e], g[e]);
          xv[j][k] = V::narrow(f);  // the residual as stored
          st_stream<VB>((char*)a.out + rowoff + coff[k], xv[j][k]);
        }
        if constexpr (kReduce) {
          V::widen(xv[j][k], f);
#pragma unroll
          for (int e = 0; e < N; ++e) {
            if constexpr (EX)
              acc.add((k * N + e) % 4, f[e]);
            else
              ssf[j] = __fmaf_rn(f[e], f[e], ssf[j]);
          }
        }
      }
      if constexpr (EX) ss[j] = acc.total();
    }
    if constexpr (kReduce) {
      // row pairs over the warp, then over the warps
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if constexpr (EX) {
          const SumPair w = warp_merge(ss[j]);
          if (lane == 0) part[buf][j][warp] = w;
        } else {
          const float w = warp_sum(ssf[j]);
          if (lane == 0) partf[buf][j][warp] = w;
        }
      }
      __syncthreads();
      float rinv[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if constexpr (!EX) {
          // the fast statistic: the warps' sums in order
          float tot = 0.0f;
          for (int w = 0; w < nwarps; ++w) tot = __fadd_rn(tot, partf[buf][j][w]);
          rinv[j] = fast_inverse_rms(tot, a.d_f, a.inv_d, a.eps);
          if (rval[j] && !fast_sum_in_range(tot)) {
            // rare, uniform over the CTA: the row's squares again, scaled
            const float sc = fast_rescale(tot);
            float s2 = 0.0f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
              if (!cval[k]) continue;
              float x[N];
              V::widen(xv[j][k], x);
#pragma unroll
              for (int e = 0; e < N; ++e) {
                const float u0 = __fmul_rn(x[e], sc);
                s2 = __fmaf_rn(u0, u0, s2);
              }
            }
            s2 = warp_sum(s2);
            if (lane == 0) part_scaled[warp] = s2;
            __syncthreads();
            float S2 = 0.0f;
            for (int w = 0; w < nwarps; ++w) S2 = __fadd_rn(S2, part_scaled[w]);
            __syncthreads();  // read before the next row's writes
            rinv[j] = fast_inverse_rms_scaled(S2, sc, a.d_f, a.inv_d, a.eps);
          }
        } else {
          const SumPair p = group_merge<16>(part[buf][j][lane & 15]);
          auto each = [=](auto&& f) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
              if (!(rval[j] && cval[k])) continue;
              float x[N];
              V::widen(xv[j][k], x);
#pragma unroll
              for (int e = 0; e < N; ++e) f(x[e]);
            }
          };
          rinv[j] = row_inverse_rms(p, coef, kLevels, a.D, a.d_f, a.eps, each,
                                    CtaRow{exact_scratch});
        }
      }
      buf ^= 1;

      void* mout = OP == OP_FUSED ? a.out2 : a.out;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int64_t rowoff = (r0 + j) * pitch;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          if (!(rval[j] && cval[k])) continue;
          float x[N], s[N], h[N], y[N];
          V::widen(xv[j][k], x);
          V::widen(MFULL ? scv[j][k] : scb[k], s);
          V::widen(MFULL ? shv[j][k] : shb[k], h);
#pragma unroll
          for (int e = 0; e < N; ++e) y[e] = modulate(x[e], rinv[j], s[e], h[e]);
          st_stream<VB>((char*)mout + rowoff + coff[k], V::narrow(y));
        }
      }
    }
  }
}

// Rows longer than one CTA can hold: two passes over each row.  The fast
// statistic keeps the compensated merge across a thread's vectors here: a
// thread may take thousands of them, and a plain fp32 running sum would then
// carry an error bound of that many units.
template <int OP, class T, int VB, bool GFULL, bool MFULL, bool EX>
__global__ void __launch_bounds__(1024) long_row_kernel(RowArgs a) {
  using V = Vec<T, VB>;
  constexpr int N = V::N;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = nthr >> 5;
  const int64_t pitch = a.D * (int64_t)sizeof(T);
  __shared__ SumPair part[2][32];        // per-warp row pairs
  __shared__ uint64_t exact_scratch[32];  // the exact path's warp totals
  for (int i = tid; i < 64; i += nthr)
    if ((i & 31) >= nwarps) (&part[0][0])[i] = SumPair{0.0f, 0.0f};
  int buf = 0;
  // the statistic: each vector's squares go through four scalar (hi, lo)
  // accumulators, then merge into the thread's running pair -- one merge
  // level per vector the thread takes
  using Acc = Sq32<4>;
  const int64_t per_thread = (a.nvec + nthr - 1) / nthr;
  [[maybe_unused]] const float coef = Acc::coef((N + 3) / 4);
  [[maybe_unused]] const int levels = (int)per_thread + 2 + 5 + 5;  // D <= 2^24

  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const int64_t b = row / a.L;
    const int64_t rowoff = row * pitch;
    const int64_t goff = GFULL ? rowoff : b * a.vstride;
    const int64_t moff = MFULL ? rowoff : b * a.vstride;
    SumPair ss{0.0f, 0.0f};
    for (int64_t v = tid; v < a.nvec; v += nthr) {
      const int64_t c = v * VB;
      float f[N];
      Raw<VB> xr = ld_stream<VB>((const char*)a.x + rowoff + c);
      if constexpr (OP == OP_FUSED) {
        float h[N], u[N], g[N];
        V::widen(xr, h);
        V::widen(ld_stream<VB>((const char*)a.u + rowoff + c), u);
        V::widen(GFULL ? ld_stream<VB>((const char*)a.g + goff + c)
                       : ld_bcast<VB>((const char*)a.g + goff + c), g);
#pragma unroll
        for (int e = 0; e < N; ++e) f[e] = residual_gate(h[e], u[e], g[e]);
        xr = V::narrow(f);
        st_stream<VB>((char*)a.out + rowoff + c, xr);
      }
      V::widen(xr, f);
      Acc acc;
      acc.zero();
#pragma unroll
      for (int e = 0; e < N; ++e) {
        if constexpr (EX)
          acc.add(e % 4, f[e]);
        else
          acc.add_fast(e % 4, f[e]);
      }
      ss = merge(ss, acc.total());
    }
    const SumPair w = warp_merge(ss);
    if (lane == 0) part[buf][warp] = w;
    __syncthreads();
    const SumPair p = warp_merge(part[buf][lane]);
    buf ^= 1;
    // each thread's vectors, read again by the exact path and the second
    // pass (for the fused op, its own residual stores)
    const void* src = OP == OP_FUSED ? (const void*)a.out : a.x;
    const int64_t nvec = a.nvec;
    auto each = [=](auto&& f) {
      for (int64_t v = tid; v < nvec; v += nthr) {
        float x[N];
        V::widen(ld_stream<VB>((const char*)src + rowoff + v * VB), x);
#pragma unroll
        for (int e = 0; e < N; ++e) f(x[e]);
      }
    };
    float rinv;
    if constexpr (EX) {
      rinv = row_inverse_rms(p, coef, levels, a.D, a.d_f, a.eps, each, CtaRow{exact_scratch});
    } else if (fast_sum_in_range(p.h) && !isnan(p.h)) {
      rinv = fast_inverse_rms(p.h, a.d_f, a.inv_d, a.eps);
    } else {
      // rare, uniform over the CTA: the row's squares again, scaled, merged
      // as pairs like the first pass.  Here a NaN sum is not only a NaN in
      // the row: the pair merges turn an infinite square into NaN (inf - inf
      // in TwoSum), so infinities are counted apart and give r = 0.
      const float sc = isnan(p.h) ? 0x1p-64f : fast_rescale(p.h);
      SumPair s2{0.0f, 0.0f};
      bool inf_seen = false;
      for (int64_t v = tid; v < nvec; v += nthr) {
        float x[N];
        V::widen(ld_stream<VB>((const char*)src + rowoff + v * VB), x);
        Acc acc;
        acc.zero();
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const bool inf = fabsf(x[e]) == __int_as_float(0x7f800000);
          inf_seen = inf_seen || inf;
          acc.add_fast(e % 4, inf ? 0.0f : __fmul_rn(x[e], sc));
        }
        s2 = merge(s2, acc.total());
      }
      const SumPair w2 = warp_merge(s2);
      if (lane == 0) part[buf][warp] = w2;
      const bool any_inf = __syncthreads_or(inf_seen) != 0;
      const SumPair p2 = warp_merge(part[buf][lane]);
      buf ^= 1;
      // a NaN in the row wins (the sum of squares is NaN), then an infinity
      rinv = isnan(p2.h) ? p2.h
                         : any_inf ? 0.0f : fast_inverse_rms_scaled(p2.h, sc, a.d_f, a.inv_d, a.eps);
    }

    // second pass: each thread re-reads exactly the vectors it handled above
    void* dst = OP == OP_FUSED ? a.out2 : a.out;
    for (int64_t v = tid; v < a.nvec; v += nthr) {
      const int64_t c = v * VB;
      float x[N], s[N], h[N], y[N];
      V::widen(ld_stream<VB>((const char*)src + rowoff + c), x);
      if constexpr (MFULL) {
        V::widen(ld_stream<VB>((const char*)a.sc + moff + c), s);
        V::widen(ld_stream<VB>((const char*)a.sh + moff + c), h);
      } else {
        V::widen(ld_bcast<VB>((const char*)a.sc + moff + c), s);
        V::widen(ld_bcast<VB>((const char*)a.sh + moff + c), h);
      }
#pragma unroll
      for (int e = 0; e < N; ++e) y[e] = modulate(x[e], rinv, s[e], h[e]);
      st_stream<VB>((char*)dst + rowoff + c, V::narrow(y));
    }
  }
}

// Rows per thread group by operation and layout: R * (streamed operands)
// * 32 bytes stays near 128 bytes in flight per thread.
// Narrow accesses (one or a few elements each) halve it: they need a
// register per access, and the tail shapes that use them are not the ones
// that set the bandwidth.
#ifndef DIT_R_RGA
#define DIT_R_RGA 2
#endif
#ifndef DIT_R_MOD
#define DIT_R_MOD 4
#endif
#ifndef DIT_R_FUSED
#define DIT_R_FUSED 2
#endif
template <int OP, bool GFULL, bool MFULL, int VB>
__host__ __device__ constexpr int rows_in_flight() {
  const int r = OP == OP_RGA   ? DIT_R_RGA
                : OP == OP_MOD ? (MFULL ? (DIT_R_MOD + 1) / 2 : DIT_R_MOD)
                               : ((GFULL || MFULL) ? (DIT_R_FUSED + 1) / 2 : DIT_R_FUSED);
  return VB >= 16 ? r : (r > 1 ? r / 2 : 1);
}

// Two-pass kernel for rows that do not fit one CTA's registers.
template <int OP, bool GFULL, bool MFULL>
cudaError_t launch_long_rows(const DeviceInfo& dev, int dtype, int vb, RowArgs a,
                             cudaStream_t stream) {
  const int64_t row_bytes = a.D * (dtype == 2 ? 4 : 2);
  // 16-byte accesses when the rows allow them, else one element at a time
  const int lvb = vb >= 16 ? 16 : (dtype == 2 ? 4 : 2);
  a.nvec = row_bytes / lvb;
  return dispatch_dtype_width(dtype, lvb, [&](auto tt, auto w) -> cudaError_t {
    using T = typename decltype(tt)::type;
    constexpr int VB = decltype(w)::value;
    if constexpr (VB == 16 || VB == (int)sizeof(T)) {
      return with_statistic<OP>(a.exact, [&](auto ex) -> cudaError_t {
        auto kern = long_row_kernel<OP, T, VB, GFULL, MFULL, decltype(ex)::value>;
        const int block = 1024;
        int64_t grid = (int64_t)dev.sm_count * resident_ctas(dev, (const void*)kern, block);
        if (grid > a.rows) grid = a.rows;
        if (grid < 1) grid = 1;
        kern<<<(unsigned)grid, block, 0, stream>>>(a);
        return cudaGetLastError();
      });
    } else {
      return cudaErrorInvalidValue;
    }
  });
}

// Whether every tensor the staged kernel streams or stores starts on a
// 16-byte boundary (the [B, 1, D] operands, read element by element in the
// phased kernel, may start anywhere).
template <int OP, bool GFULL, bool MFULL>
bool streamed_bases_aligned(const RowArgs& a) {
  uintptr_t bits = (uintptr_t)a.out | (uintptr_t)a.x;
  if (OP != OP_MOD) bits |= (uintptr_t)a.u;
  if (OP != OP_MOD && GFULL) bits |= (uintptr_t)a.g;
  if (OP != OP_RGA && MFULL) bits |= (uintptr_t)a.sc | (uintptr_t)a.sh;
  if (OP == OP_FUSED) bits |= (uintptr_t)a.out2;
  return (bits & 15u) == 0;
}

// Rows aligned to 16 bytes take the shared-memory-staged kernel (dit_pipe.cuh);
// rows of other pitches whose tensors start on 16-byte boundaries take it by
// phase -- except the reducing operations on 8-byte aligned rows, where the
// register kernel's 8-byte accesses were as fast or faster (L2-flushed,
// [1,4097,3076] bf16: modulation 22.4 vs 22.7 us, fused 33.2 vs 36.8 us; the
// residual gate 20.1 vs 20.5 us phased); other narrow alignments the
// register-resident row kernel; rows too long for one CTA the two-pass kernel.
template <int OP, bool GFULL, bool MFULL>
cudaError_t launch_row_op(const DeviceInfo& dev, int dtype, int vb, RowArgs a, int64_t B,
                          cudaStream_t stream) {
  const int64_t row_bytes = a.D * (dtype == 2 ? 4 : 2);
#ifndef DIT_ROWS_IN_REGISTERS
  if constexpr (OP != OP_RGA && !GFULL && !MFULL) {
    // the modulating ops on rows of other pitches in 16-byte aligned tensors,
    // with the fast statistic: two warps per row, by phase
    if (vb < 16 && !a.exact && streamed_bases_aligned<OP, GFULL, MFULL>(a)) {
      const cudaError_t w =
          launch_wrow<OP, GFULL, MFULL, false, false>(dev, dtype, a, B, stream, true);
      if (w != cudaErrorNotSupported) return w;
    }
  }
  if (vb < 16 && (OP == OP_RGA || vb < 8) && streamed_bases_aligned<OP, GFULL, MFULL>(a)) {
    const cudaError_t e = with_statistic<OP>(a.exact, [&](auto ex) {
      return launch_pipe<OP, GFULL, MFULL, false, decltype(ex)::value>(dev, dtype, a, B, stream,
                                                                        true);
    });
    if (e != cudaErrorNotSupported) return e;
  }
#endif
#ifdef DIT_ROWS_IN_REGISTERS  // tuning builds: the register kernel for every width
  if (false) {
#else
  if (vb >= 16) {
#endif
    // two warps per row (dit_wrow.cuh) when the row fits their registers;
    // not for the fused op with a full gate: a third staged operand (96 KB of
    // stages) leaves one CTA per SM, and the CTA-per-row kernel was faster
    // ([1,8160,4096] bf16, L2-flushed: 53.8 vs 65.9 us)
    if constexpr (OP != OP_RGA && !(OP == OP_FUSED && GFULL)) {
      const cudaError_t w = with_statistic<OP>(a.exact, [&](auto ex) {
        return launch_wrow<OP, GFULL, MFULL, false, decltype(ex)::value>(dev, dtype, a, B, stream);
      });
      if (w != cudaErrorNotSupported) return w;
    }
    const cudaError_t e = with_statistic<OP>(a.exact, [&](auto ex) {
      return launch_pipe<OP, GFULL, MFULL, false, decltype(ex)::value>(dev, dtype, a, B, stream);
    });
    if (e != cudaErrorNotSupported) return e;
    if constexpr (OP == OP_RGA) {
      return cudaErrorInvalidValue;  // unreachable: the residual gate tiles columns
    } else {
      return launch_long_rows<OP, GFULL, MFULL>(dev, dtype, vb, a, stream);
    }
  }
  a.nvec = row_bytes / vb;
  bool too_long = false;
  const cudaError_t e = dispatch_dtype_width(dtype, vb, [&](auto tt, auto w) -> cudaError_t {
    using T = typename decltype(tt)::type;
    constexpr int VB = decltype(w)::value;
#ifdef DIT_ROWS_IN_REGISTERS
    if constexpr (false) {
#else
    if constexpr (VB >= 16) {
#endif
      return cudaErrorInvalidValue;  // handled by the staged kernel above
    } else {
    constexpr int TB = thread_bytes<VB>();
    constexpr int R = rows_in_flight<OP, GFULL, MFULL, VB>();
    const int64_t threads_needed = (row_bytes + TB - 1) / TB;
    return with_statistic<OP>(a.exact, [&](auto ex) -> cudaError_t {
    auto kern = row_kernel<OP, T, VB, R, GFULL, MFULL, decltype(ex)::value>;
    const void* fn = (const void*)kern;
    int block;
    unsigned slices = 1;
    if (OP == OP_RGA) {
      // equal column slices of at most kRowBlockMax threads
      const int64_t s = (threads_needed + kRowBlockMax - 1) / kRowBlockMax;
      if (s > 65535) return cudaErrorInvalidConfiguration;
      slices = (unsigned)s;
      block = (int)(((threads_needed + s - 1) / s + 31) / 32 * 32);
    } else {
      if (threads_needed > kRowBlockMax) {
        too_long = true;
        return cudaSuccess;
      }
      block = (int)((threads_needed + 31) / 32 * 32);
    }
    a.gpb = (a.L + R - 1) / R;
    a.ngroups = B * a.gpb;
    int64_t G = (int64_t)dev.sm_count * resident_ctas(dev, fn, block);
    if (G > a.ngroups) G = a.ngroups;
    if (G < 1) G = 1;
    if (G > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    a.step_b = G / a.gpb;
    a.step_g = G - a.step_b * a.gpb;
    kern<<<dim3((unsigned)G, slices, 1), dim3((unsigned)block, 1, 1), 0, stream>>>(a);
    return cudaGetLastError();
    });
    }
  });
  if (e != cudaSuccess || !too_long) return e;
  if constexpr (OP == OP_RGA) {
    return cudaErrorInvalidValue;  // unreachable: the residual gate tiles columns
  } else {
    return launch_long_rows<OP, GFULL, MFULL>(dev, dtype, vb, a, stream);
  }
}

}  // namespace dit
