// dit_wrow.cuh -- the modulation and the fused op with two warps per row
// (sm_103a; rows of up to 8 KB in 16-byte aligned tensors, whose pitch is a
// multiple of 16 bytes -- or any pitch, by phase, with the fast statistic).
//
// A row belongs to a team of two warps; lane l of member m holds 16-byte
// granules l + 32 m + 64 j, j < NG, in registers, so every warp-wide access is
// 512 contiguous bytes.  The row statistic (dit_stat.cuh) is merged with warp
// shuffles and one exchange between the two warps (a 64-thread named
// barrier) -- no CTA barrier -- and its per-row work (pair merges, the
// rounding of the mean, the inverse root) runs in the two warps of the row,
// where a CTA spanning the row repeats it in each of its warps.  Two warps per
// row halve the registers that hold the row (more warps resident per SM to
// cover latency) and the time a warp spends on a row (a shorter tail).
//
// Prefetch.  Each warp owns a stage in shared memory holding its half of one
// row of the streamed inputs (x; or hidden, update and a full gate).  Each
// lane copies the granules it will read itself (cp.async), so
// cp.async.wait_group -- a hardware wait, no spin -- is the only
// synchronisation the stage needs.  The copy of the team's next row is issued
// as soon as the current row has been read out of the stage (after pass one,
// or after the fused op's residual), so it is in flight while the warp
// finishes the row.  A full scale and shift (per-token modulation) are read
// straight from global memory in pass two.
//
// The [B, 1, D] operands of the CTA's batch live in shared memory as fp32 --
// gate, 1 + scale (formed once, one fp32 rounding, as the definition has it)
// and shift -- in planes of four columns: plane q of granule g holds columns
// g * EPG + 4q .. + 3, so a warp's 16-byte reads of one plane are 512
// contiguous bytes (no bank conflicts).
//
// Schedule.  On large tensors (more than 8 rows per team in one wave of
// CTAs) a CTA gives each of its teams a few rows (three for the modulation,
// two for the fused op) of one batch, and the grid holds as many CTAs as that
// takes -- several waves, handed to the SMs by the hardware as earlier CTAs
// finish.  With the fast statistic the last wave of each batch's CTAs takes
// one row per team: an SM whose last long CTA ends early picks these up, so
// the SMs finish within about one row of each other instead of three (ncu,
// modulation of [1,32640,4096] bf16: active cycles per SM 146k-166k without
// the tail, 148k-156k with it).  A one-wave persistent grid, each CTA
// striding over the tensor, left SMs idle at the end there: the SMs do not stream at the same rate,
// and a static split of the rows made the slowest SM set the kernel's length
// (on [1,32640,4096] bf16 the modulation took 98 us back to back with it, 86
// us with four rows per team, 84 with three -- 1, 2, 6 and 8 were slower, as
// were 12-warp CTAs; the fused op 182 and 160 us with two).  Smaller
// tensors run exactly one wave with the rows split statically: there a
// second, partial wave of short CTAs costs more than the imbalance
// ([1,8160,4096]: 510 CTAs of four rows per team, 1.1 waves, ran the
// modulation in 35.7 us L2-flushed).  Of a batch's CTAs the first H (the
// head) give their team t rows k * T + t, k * T + t + H * T, ... of the
// batch's first head_rows rows (T teams per CTA; without a tail H is all of
// them and head_rows the whole batch); tail CTA k gives team t the one row
// head_rows + (k - H) * T + t.  The grid is capped at 64 waves; with more
// batches than that a CTA takes batches c, c + grid, ..., reloading the
// vectors (two barriers) between them, and there is no tail.
#pragma once

#include <algorithm>
#include <atomic>

#include "dit_device.cuh"
#include "dit_internal.h"
#include "dit_pipe.cuh"
#include "dit_stat.cuh"

namespace dit {

constexpr int kWrowWarps = 8;  // warps per CTA: four teams of two

// [B, 1, D] vectors held in shared memory, and operands staged per row.
template <int OP, bool GFULL, bool MFULL>
__host__ __device__ constexpr int wrow_vectors() {
  return (OP == OP_FUSED && !GFULL ? 1 : 0) + (MFULL ? 0 : 2);
}
template <int OP, bool GFULL>
__host__ __device__ constexpr int wrow_staged() {
  return OP == OP_MOD ? 1 : (GFULL ? 3 : 2);
}

// CTAs per SM the register bound is set for: the modulation three 8-warp
// CTAs (at most 85 registers) and the fused op two (128), with up to 8
// granules per lane; rows of 12 or 16 granules per lane one fewer.
template <int OP, int NG>
constexpr int wrow_min_blocks() {
  return (OP == OP_FUSED ? 2 : 3) - (NG > 8 ? 1 : 0);
}

// The two warps of a row, for the exact paths of the statistic: a warp
// reduction, then the two warps' values through shared memory between two
// 64-thread named barriers (id 1 + team).
struct TeamRow {
  uint64_t* xch;  // two words of this team
  int id, m;
  __device__ __forceinline__ uint64_t both(uint64_t v, bool add, bool take_min) const {
    if ((threadIdx.x & 31) == 0) xch[m] = v;
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
    const uint64_t a = xch[0], b = xch[1];
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
    return add ? a + b : take_min ? (a < b ? a : b) : (a > b ? a : b);
  }
  __device__ __forceinline__ uint64_t sum(uint64_t v) const { return both(WarpRow().sum(v), true, false); }
  __device__ __forceinline__ int imin(int v) const {
    return (int)both((uint64_t)(int64_t)(WarpRow().imin(v) + 1), false, true) - 1;
  }
  __device__ __forceinline__ int imax(int v) const {
    return (int)both((uint64_t)(int64_t)(WarpRow().imax(v) + 1), false, false) - 1;
  }
  __device__ __forceinline__ bool any(bool b) const {
    return both(WarpRow().any(b) ? 1u : 0u, false, false) != 0u;
  }
};

// EX: the exact row statistic (dit_set_statistic); otherwise the fast one.
// Each is its own instantiation, so the fast kernel carries none of the
// exact path's registers.
//
// PH (phased rows; the fast statistic, [B, 1, D] operands only): the row
// pitch is not a multiple of 16 bytes but every streamed tensor starts on a
// 16-byte boundary.  Row r then starts (r * pitch) mod 16 bytes past a
// boundary, a value of period P = 16 / gcd(pitch mod 16, 16) rows, so the
// CTAs of a batch are split into P phase classes: class c takes rows
// c, c + P, c + 2P, ..., all at one offset `off`.  A team copies a row's
// 16-byte granules from the boundary below its start (the last row's last
// granule only up to the tensors' end); a row's first and last granule hold
// elements of its neighbours, masked out of the sum and never stored (the
// row's own elements of them are stored one by one).  The CTA's vector
// planes are written at the same offset, so granule k of the window meets
// the vector columns of its elements.
template <int OP, class T, int NG, bool GFULL, bool MFULL, bool Q8, bool EX, bool PH = false>
__global__ void __launch_bounds__(kWrowWarps * 32, wrow_min_blocks<OP, NG>()) wrow_kernel(RowArgs a) {
  using G = Granule<T>;
  constexpr int P = G::P;     // fp32 pairs per granule
  constexpr int NPL = P / 2;  // planes of four columns per granule
  constexpr int NV = wrow_vectors<OP, GFULL, MFULL>();
  constexpr int NS = wrow_staged<OP, GFULL>();
  constexpr bool kGateV = OP == OP_FUSED && !GFULL;
  // the statistic: 4 packed slots, granule j's pair i in slot (j % R) * P + i
  constexpr int kNA = 4;
  constexpr int R = kNA / P;
  using Acc = SqAcc<T, kNA>;
  constexpr int kTerms = (NG + R - 1) / R;
  constexpr int kLevels = Log2<Acc::kScalar>::value + 5 + 1;  // thread, warp, team
  constexpr uint32_t kStage = NG * 512;  // bytes of one staged operand per warp
  constexpr int ES = (int)sizeof(T);
  constexpr int EPG = 16 / ES;  // elements per granule
  static_assert(!PH || (!EX && !Q8 && !MFULL && !GFULL), "phased rows: fast statistic, [B,1,D]");

  extern __shared__ float4 vsm[];  // [NV][NPL][ngr] vectors, then [W][NS][NG * 32] stages
  __shared__ SumPair xch_pair[2][kWrowWarps / 2][2];  // the team's pair exchange, by row parity
  __shared__ uint64_t xch_exact[kWrowWarps / 2][2];
  __shared__ float xch_scaled[kWrowWarps / 2][2];  // the fast statistic's rescaled sums
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = warp >> 1, m = warp & 1;
  const int nteams = blockDim.x >> 6;
  const int64_t ngr = a.nvec;  // granules per row (phased: at most, over the offsets)
  const uint32_t pls = (uint32_t)ngr * 16;  // bytes per vector plane
  // this lane's granules: l + 32 m + 64 j
  const uint32_t lg = (uint32_t)(lane + 32 * m);
  bool val[NG];
#pragma unroll
  for (int j = 0; j < NG; ++j) val[j] = lg + 64 * j < ngr;
  const float coef = Acc::coef(kTerms);

  // shared addresses of this lane's granule 0 (granule j: + j * 1024): one
  // base per vector plane and per staged operand
  const uint32_t vbase = smem_addr(vsm) + lg * 16;
  uint32_t gvs[NPL], onev[NPL], shv[NPL], stage[3];
#pragma unroll
  for (int q = 0; q < NPL; ++q) {
    gvs[q] = vbase + q * pls;
    onev[q] = vbase + ((kGateV ? NPL : 0) + q) * pls;
    shv[q] = vbase + ((kGateV ? NPL : 0) + NPL + q) * pls;
  }
  const uint32_t sbase = smem_addr(vsm) + NV * NPL * pls + (uint32_t)warp * NS * kStage + lane * 16;
#pragma unroll
  for (int op = 0; op < 3; ++op) stage[op] = sbase + op * kStage;
  const char* const src[3] = {(const char*)a.x, (const char*)a.u, (const char*)a.g};
  const TeamRow trow{&xch_exact[team][0], 1 + team, m};

  // batches: a.gpb = CTAs per batch, a.ngroups = batches served at once
  const int64_t cpb = a.gpb;
  const int64_t slot = (int64_t)blockIdx.x / cpb, kc = (int64_t)blockIdx.x - slot * cpb;
  const int64_t nbatch = a.rows / (a.L > 0 ? a.L : 1);
  const int64_t pitch = a.D * (int64_t)ES;
  // phased rows: this CTA's phase class c of the period (cpb is a multiple
  // of it), kq its index among the class's CTAs
  int64_t period = 1;
  if constexpr (PH) {
    const int64_t mm = pitch & 15;
    period = mm ? 16 / (mm & -mm) : 1;
  }
  const int64_t phase = kc % period, kq = kc / period;
  const int64_t rstep = cpb * nteams;  // = period * (cpb / period) * nteams
  float qinv_s = 1.0f;
  if constexpr (Q8) qinv_s = __frcp_rn(__ldg(a.qscale));
  const F2 qinv = f2(qinv_s, qinv_s);
  constexpr int QB = 16 / (int)sizeof(T);  // E4M3 bytes per granule
  int par = 0;

  for (int64_t b = slot; b < nbatch; b += a.ngroups) {
    // phased rows: the offset of this CTA's rows past a 16-byte boundary,
    // the granules of a row's window, and this lane's edge bounds (element
    // slots [lo, hi) of a granule belong to the row)
    int off = 0;
    int64_t ngw = ngr;
    if constexpr (PH) {
      off = (int)(((b * a.L + phase) * pitch) & 15);
      ngw = (off + pitch + 15) >> 4;
#pragma unroll
      for (int j = 0; j < NG; ++j) val[j] = lg + 64 * j < ngw;
    }
    // (only granule 0 and granule ngw - 1 of a row are partial: this lane
    // owns the first when lg == 0, the last as its granule last_j)
    [[maybe_unused]] const bool first = PH && lg == 0;
    [[maybe_unused]] const int last_j = PH && (ngw - 1) % 64 == lg ? (int)((ngw - 1) / 64) : -1;
    [[maybe_unused]] const int lo_first = off / ES;
    [[maybe_unused]] const int hi_last = (int)((off + pitch - 16 * (ngw - 1)) / ES);
    auto edge = [&](int j) { return PH && ((j == 0 && first) || j == last_j); };
    auto lo_of = [&](int j) { return j == 0 && first ? lo_first : 0; };
    auto hi_of = [&](int j) { return j == last_j ? hi_last : EPG; };

    // this team's rows of the batch: l, l + lstep, ... below lend -- a head
    // CTA (kc < a.step_b) strides over rows [0, a.step_g), a tail CTA takes
    // one row of the rest (phased rows: the CTA's phase class, over the
    // whole batch)
    int64_t l, lend = a.L, lstep = rstep;
    if constexpr (PH) {
      l = phase + period * (kq * nteams + team);
    } else if (kc < a.step_b) {
      l = kc * nteams + team;
      lend = a.step_g;
      lstep = a.step_b * nteams;
    } else {
      l = a.step_g + (kc - a.step_b) * nteams + team;
      lstep = a.L;
    }

    // copy this warp's half of row l into the stage (an empty group past the end)
    auto prefetch = [&](int64_t l) {
      if (l < lend) {
        const int64_t row = b * a.L + l;
        const int64_t rowoff = row * pitch - off + lg * 16;
        // phased rows: the last row's last granule may run past the end
        const bool tail = PH && row == a.rows - 1;
#pragma unroll
        for (int op = 0; op < NS; ++op)
#pragma unroll
          for (int j = 0; j < NG; ++j) {
            if (!val[j]) continue;
            if (tail) {
              const int64_t left = a.rows * pitch - (rowoff + j * 1024);
              if (left < 16) {
                cp_async16_part(stage[op] + j * 512, src[op] + rowoff + j * 1024, (uint32_t)left);
                continue;
              }
            }
            cp_async16(stage[op] + j * 512, src[op] + rowoff + j * 1024);
          }
      }
      cp_async_commit();
    };

    prefetch(l);  // in flight while the vectors load
    if constexpr (NV > 0) {
      __syncthreads();  // the previous batch's vectors are no longer read
      for (int64_t g = threadIdx.x; g < ngw; g += blockDim.x) {
        const int64_t vo = b * a.vstride + g * 16;
        int v = 0;
        auto put = [&](const void* vsrc, bool plus_one) {
          F2 f[P];
          if constexpr (PH) {
            // element by element, at the rows' offset (slots outside the row: 0)
            const int64_t e0 = (g * 16 - off) / ES;  // the row element at slot 0
            float e[EPG];
#pragma unroll
            for (int i = 0; i < EPG; ++i) {
              e[i] = 0.0f;
              if (e0 + i >= 0 && e0 + i < a.D) {
                float w[1];
                Vec<T, ES>::widen(ld_bcast<ES>((const char*)vsrc + b * a.vstride + (e0 + i) * ES), w);
                e[i] = w[0];
              }
            }
#pragma unroll
            for (int i = 0; i < P; ++i) f[i] = f2(e[2 * i], e[2 * i + 1]);
          } else {
            G::widen(ld_bcast<16>((const char*)vsrc + vo), f);
          }
          if (plus_one) {
#pragma unroll
            for (int i = 0; i < P; ++i) f[i] = f2_add(f2(1.0f, 1.0f), f[i]);
          }
#pragma unroll
          for (int q = 0; q < NPL; ++q)
            vsm[((int64_t)v * NPL + q) * ngr + g] =
                make_float4(f2_lo(f[2 * q]), f2_hi(f[2 * q]), f2_lo(f[2 * q + 1]), f2_hi(f[2 * q + 1]));
          ++v;
        };
        if constexpr (kGateV) put(a.g, false);
        if constexpr (!MFULL) {
          put(a.sc, true);
          put(a.sh, false);
        }
      }
      __syncthreads();
    }

    for (; l < lend; l += lstep) {
      const int64_t row = b * a.L + l;
      const int64_t rowoff = row * pitch - off + lg * 16;
      cp_async_wait<0>();  // this lane's copies of row l have landed
      Raw<16> xr[NG];
      if constexpr (OP == OP_FUSED) {
        // the residual: hidden + update * gate, rounded, stored, kept
        char* const res = (char*)a.out + rowoff;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          if (!val[j]) continue;
          F2 h[P], u[P], g[P], x[P];
          G::widen(lds16(stage[0] + j * 512), h);
          G::widen(lds16(stage[1] + j * 512), u);
          if constexpr (GFULL) {
            G::widen(lds16(stage[2] + j * 512), g);
          } else {
#pragma unroll
            for (int q = 0; q < NPL; ++q) {
              const Raw<16> v = lds16(gvs[q] + j * 1024);
              g[2 * q] = f2(__uint_as_float(v.w[0]), __uint_as_float(v.w[1]));
              g[2 * q + 1] = f2(__uint_as_float(v.w[2]), __uint_as_float(v.w[3]));
            }
          }
#pragma unroll
          for (int i = 0; i < P; ++i) x[i] = residual_gate2<T>(h[i], u[i], g[i]);
          xr[j] = G::narrow(x);
          if (edge(j))
            store_part<T>(res + j * 1024, xr[j], lo_of(j), hi_of(j));
          else
            st_stream<16>(res + j * 1024, xr[j]);
        }
        prefetch(l + lstep);  // the stage has been read
      } else {
#pragma unroll
        for (int j = 0; j < NG; ++j)
          if (val[j]) xr[j] = lds16(stage[0] + j * 512);
      }

      // pass one and the statistic (the exact one or the fast one); the
      // stage's next copy is issued once xr is read out
      float r;
      if constexpr (EX) {
        Acc acc;
        acc.zero();
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          if (!val[j]) continue;
          F2 x[P];
          G::widen(xr[j], x);
#pragma unroll
          for (int i = 0; i < P; ++i) acc.add_pair((j % R) * P + i, x[i]);
        }
        if constexpr (OP != OP_FUSED) prefetch(l + lstep);
        SumPair p = warp_merge(acc.total());
        // the other warp of the row: exchange through shared memory (one
        // slot pair per row parity, so a slot is rewritten only after the
        // next barrier, which the other warp reaches after reading it)
        if (lane == 0) xch_pair[par][team][m] = p;
        asm volatile("bar.sync %0, 64;" ::"r"(1 + team) : "memory");
        p = merge(p, xch_pair[par][team][m ^ 1]);
        // the exact paths read the lane's granules back from global memory
        // (x, or the residual this lane stored): nothing of the hot path's
        // registers is captured, and the loop is not unrolled
        const char* const back = (OP == OP_FUSED ? (const char*)a.out : (const char*)a.x) + rowoff;
        auto each = [=](auto&& f) {
#pragma unroll 1
          for (int j = 0; j < NG; ++j) {
            if (lg + 64 * j >= ngr) continue;
            F2 x[P];
            G::widen(ld_stream<16>(back + j * 1024), x);
#pragma unroll
            for (int i = 0; i < P; ++i) {
              f(f2_lo(x[i]));
              f(f2_hi(x[i]));
            }
          }
        };
        r = row_inverse_rms(p, coef, kLevels, a.D, a.d_f, a.eps, each, trow);
      } else {
        Acc acc;
        acc.zero();
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          if (!val[j]) continue;
          F2 x[P];
          G::widen(xr[j], x);
          if (edge(j)) mask_part<T>(x, lo_of(j), hi_of(j));
#pragma unroll
          for (int i = 0; i < P; ++i) acc.add_pair_fast((j % R) * P + i, x[i]);
        }
        if constexpr (OP != OP_FUSED) prefetch(l + lstep);
        const float ws = warp_sum(acc.fast_total());
        if (lane == 0) xch_pair[par][team][m] = SumPair{ws, 0.0f};
        asm volatile("bar.sync %0, 64;" ::"r"(1 + team) : "memory");
        // both warps add the two halves in the same order
        const float S = __fadd_rn(xch_pair[par][team][0].h, xch_pair[par][team][1].h);
        if (fast_sum_in_range(S)) {
          r = fast_inverse_rms(S, a.d_f, a.inv_d, a.eps);
        } else {
          // rare (both warps of the team): the squares of the row scaled
          const float sc = fast_rescale(S);
          float s2 = 0.0f;
#pragma unroll
          for (int j = 0; j < NG; ++j) {
            if (!val[j]) continue;
            F2 x[P];
            G::widen(xr[j], x);
            if (edge(j)) mask_part<T>(x, lo_of(j), hi_of(j));
#pragma unroll
            for (int i = 0; i < P; ++i) {
              const float u0 = __fmul_rn(f2_lo(x[i]), sc), u1 = __fmul_rn(f2_hi(x[i]), sc);
              s2 = __fmaf_rn(u1, u1, __fmaf_rn(u0, u0, s2));
            }
          }
          s2 = warp_sum(s2);
          if (lane == 0) xch_scaled[team][m] = s2;
          asm volatile("bar.sync %0, 64;" ::"r"(1 + team) : "memory");
          const float S2 = __fadd_rn(xch_scaled[team][0], xch_scaled[team][1]);
          asm volatile("bar.sync %0, 64;" ::"r"(1 + team) : "memory");  // read before reuse
          r = fast_inverse_rms_scaled(S2, sc, a.d_f, a.inv_d, a.eps);
        }
      }
      par ^= 1;
      const F2 r2 = f2(r, r);

      // pass two: normalise, modulate, store
      char* const mout = (char*)(OP == OP_FUSED ? a.out2 : a.out) + (Q8 ? row * a.D + lg * QB : rowoff);
      const char* const scr = (const char*)a.sc + rowoff;
      const char* const shr = (const char*)a.sh + rowoff;
#pragma unroll
      for (int j = 0; j < NG; ++j) {
        if (!val[j]) continue;
        F2 x[P], one[P], sh[P], y[P];
        G::widen(xr[j], x);
        if constexpr (MFULL) {
          G::widen(ld_stream<16>(scr + j * 1024), one);
#pragma unroll
          for (int i = 0; i < P; ++i) one[i] = f2_add(f2(1.0f, 1.0f), one[i]);
          G::widen(ld_stream<16>(shr + j * 1024), sh);
        } else {
#pragma unroll
          for (int q = 0; q < NPL; ++q) {
            const Raw<16> o = lds16(onev[q] + j * 1024), s = lds16(shv[q] + j * 1024);
            one[2 * q] = f2(__uint_as_float(o.w[0]), __uint_as_float(o.w[1]));
            one[2 * q + 1] = f2(__uint_as_float(o.w[2]), __uint_as_float(o.w[3]));
            sh[2 * q] = f2(__uint_as_float(s.w[0]), __uint_as_float(s.w[1]));
            sh[2 * q + 1] = f2(__uint_as_float(s.w[2]), __uint_as_float(s.w[3]));
          }
        }
#pragma unroll
        for (int i = 0; i < P; ++i) y[i] = modulate2(f2_mul(x[i], r2), one[i], sh[i]);
        if constexpr (Q8)
          st_stream<2 * P>(mout + j * 64 * QB, quantise_e4m3<P>(y, qinv));
        else if (edge(j))
          store_part<T>(mout + j * 1024, G::narrow(y), lo_of(j), hi_of(j));
        else
          st_stream<16>(mout + j * 1024, G::narrow(y));
      }
    }
    cp_async_wait<0>();  // the last (empty) group: nothing outlives the batch
  }
}

// Granules per lane of the instantiated kernels: 2, 4, 8 (a row of n
// granules takes the smallest NG >= n / 64): rows up to 8 KB.  Longer rows
// take the CTA-per-row kernel: with 12 granules per lane the fused op needed
// 244 registers (one CTA per SM) and the modulation 126 (two), and both ran
// slower than the CTA-per-row kernel on [1,4096,4608] bf16.
constexpr int kWrowMaxNG = 8;

// Tenths of a wave of one-row-per-team CTAs that end each batch's CTAs on
// large tensors.  [1,32640,4096] bf16 back to back, modulation: none 84.3 us,
// half a wave 82.0, one wave 82.2, one and a half 82.3, two and a half 82.7;
// the fused op 158.9 against 157.8-158.2 (0.5 to 1.2 waves).
constexpr int kWrowTaper = 10;

// Launch the two-warps-per-row kernel; cudaErrorNotSupported when the row
// does not fit it (more than 64 * kWrowMaxNG granules, or the stages and the
// vectors do not fit shared memory) -- the caller then takes the CTA-per-row
// kernel.
// phased: rows whose pitch is not a multiple of 16 bytes, every streamed
// tensor 16-byte aligned (the fast statistic and [B, 1, D] operands only;
// cudaErrorNotSupported otherwise).
template <int OP, bool GFULL, bool MFULL, bool Q8, bool EX>
cudaError_t launch_wrow(const DeviceInfo& dev, int dtype, RowArgs a, int64_t B,
                        cudaStream_t stream, bool phased = false) {
  constexpr bool kPhasedOk = !EX && !Q8 && !MFULL && !GFULL;
  if (phased && !kPhasedOk) return cudaErrorNotSupported;
  const int64_t row_bytes = a.D * (dtype == 2 ? 4 : 2);
  // granules per row (phased: at most, over the rows' offsets)
  a.nvec = phased ? (row_bytes + 30) / 16 : row_bytes / 16;
  const int64_t mm = row_bytes & 15;
  const int64_t period = phased && mm ? 16 / (mm & -mm) : 1;
  const int64_t need = (a.nvec + 63) / 64;
  if (need > kWrowMaxNG) return cudaErrorNotSupported;
  static_assert(!(OP == OP_FUSED && GFULL), "the fused op with a full gate is not instantiated");
  constexpr int NV = wrow_vectors<OP, GFULL, MFULL>();
  constexpr int NS = wrow_staged<OP, GFULL>();
  const size_t vbytes = (size_t)NV * (size_t)a.nvec * 16 * (dtype == 2 ? 1 : 2);
  const size_t limit = (size_t)(dev.smem_optin - kStaticSmemReserve);
  return dispatch_dtype_width(dtype, 16, [&](auto tt, auto) -> cudaError_t {
    using T = typename decltype(tt)::type;
    auto go = [&](auto ng) -> cudaError_t {
      constexpr int NG = decltype(ng)::value;
      auto kern = wrow_kernel<OP, T, NG, GFULL, MFULL, Q8, EX, false>;
      if constexpr (kPhasedOk)
        if (phased) kern = wrow_kernel<OP, T, NG, GFULL, MFULL, Q8, EX, true>;
      const size_t smem = vbytes + (size_t)kWrowWarps * NS * NG * 512;
      if (smem > limit) return cudaErrorNotSupported;
      // one opt-in record per kernel (the phased kernel is another function)
      static std::atomic<int> opted_plain[kOptinDevices], opted_phased[kOptinDevices];
      const cudaError_t e =
          allow_dynamic_smem((const void*)kern, dev, smem, phased ? opted_phased : opted_plain);
      if (e != cudaSuccess) return e;
      const int block = kWrowWarps * 32;
      const int teams = kWrowWarps / 2;
      // short-lived CTAs of a few rows per team, handed to SMs by the
      // hardware as they free up, and at least one wave of them when the
      // rows allow (one row per team at least)
      const int64_t wave = (int64_t)dev.sm_count * resident_ctas(dev, (const void*)kern, block, smem);
      const int64_t most = (a.L + teams - 1) / teams;  // CTAs per batch, one row per team
      int64_t per_batch;
      const bool small = B * a.L <= 8 * wave * teams;
      // all CTAs stride over the whole batch, unless tapered below
      int64_t head = -1, head_rows = a.L;
      // the fused op takes this kernel on large tensors only: on smaller ones
      // the CTA-per-row kernel, with three CTAs per SM to its two, was faster
      // ([1,4608,3072] bf16, L2-flushed: 25.3 vs 27.1 us)
      if (OP == OP_FUSED && small && !phased) return cudaErrorNotSupported;
      if (small) {
        // at most 8 rows per team in one wave: exactly one wave (fewer rows
        // than teams: one row per team), the rows split statically
        per_batch = std::min(most, (wave + B - 1) / B);
      } else {
        const int64_t rows_per_team = OP == OP_FUSED ? 2 : 3;
        per_batch = (a.L + teams * rows_per_team - 1) / (teams * rows_per_team);
        if (!phased && !EX) {
          // tapered: the last kWrowTaper / 10 waves of CTAs (over all
          // batches) take one row per team, so the SMs finish together.  Not
          // under the exact statistic, whose kernels are issue-bound rather
          // than held up by the tail (the hot-path step's exact modulation
          // 112.2 us with the tail, 112.3 without)
          const int64_t tail_ctas = (kWrowTaper * wave / 10 + B - 1) / B;  // per batch
          const int64_t tail_rows = std::min(a.L, tail_ctas * teams);
          head_rows = a.L - tail_rows;
          head = (head_rows + teams * rows_per_team - 1) / (teams * rows_per_team);
          per_batch = head + (tail_rows + teams - 1) / teams;
        }
      }
      per_batch = (per_batch + period - 1) / period * period;  // whole phase classes
      int64_t G = B * per_batch;
      if (G > 64 * wave) G = 64 * wave;  // very many batches: CTAs stride over them
      if (G < 1) G = 1;
      const int64_t nb = B < G ? B : G;  // batches served at once
      int64_t cpb = G / nb / period * period;  // CTAs per batch, a multiple of the period
      if (cpb < period) cpb = period;
      a.gpb = cpb;
      a.ngroups = nb;
      const bool tapered = head >= 0 && nb == B && cpb == per_batch;
      a.step_b = tapered ? head : cpb;
      a.step_g = tapered ? head_rows : a.L;
      const int64_t grid = nb * cpb;
      if (grid > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
      kern<<<(unsigned)grid, block, smem, stream>>>(a);
      return cudaGetLastError();
    };
    if (need <= 2) return go(std::integral_constant<int, 2>{});
    if (need <= 4) return go(std::integral_constant<int, 4>{});
    return go(std::integral_constant<int, 8>{});
  });
}

// Instantiated once, in k_instances.cu.
#define DIT_WROW_SIG(o, g, m, q, e)                                                       \
  template cudaError_t launch_wrow<o, g, m, q, e>(const DeviceInfo&, int, RowArgs, int64_t, \
                                                  cudaStream_t, bool)
extern DIT_WROW_SIG(OP_MOD, false, false, false, false);
extern DIT_WROW_SIG(OP_MOD, false, true, false, false);
extern DIT_WROW_SIG(OP_FUSED, false, false, false, false);
extern DIT_WROW_SIG(OP_FUSED, false, true, false, false);
extern DIT_WROW_SIG(OP_MOD, false, false, false, true);
extern DIT_WROW_SIG(OP_MOD, false, true, false, true);
extern DIT_WROW_SIG(OP_FUSED, false, false, false, true);
extern DIT_WROW_SIG(OP_FUSED, false, true, false, true);
extern DIT_WROW_SIG(OP_MOD, false, false, true, true);
extern DIT_WROW_SIG(OP_MOD, false, true, true, true);
extern DIT_WROW_SIG(OP_FUSED, false, false, true, true);
extern DIT_WROW_SIG(OP_FUSED, false, true, true, true);

}  // namespace dit
