// dit_pipe.cuh -- shared-memory-staged row kernels (16-byte aligned rows, and
// by phase rows of any pitch in 16-byte aligned tensors).
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
// Schedule: rows are taken in groups of RC (never straddling a batch), and
// CTA c of G takes groups c, c + G, c + 2G, ...: at any moment the G CTAs
// stream one contiguous window of the tensors, as a flat grid-stride loop
// would, instead of G scattered chunks.
//
// The [B, 1, D] operands are loaded per CTA (again only when its batch
// changes) and kept in registers in
// fp32, with 1 + scale already formed (one fp32 rounding, as in the
// modulation's definition).  The modulation takes two passes over the staged
// row: sum of squares, then -- after the reduction -- normalise, modulate and
// store.  The fused op computes the residual in pass one, stores it to HBM,
// writes it back over its own hidden slot, and pass two reads it from there.
#pragma once

#include <atomic>
#include <type_traits>

#include "dit_device.cuh"
#include "dit_internal.h"
#include "dit_stat.cuh"

namespace dit {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// the first `bytes` bytes of a 16-byte granule, the rest of the slot zeroed
// (the last granule of a phased tensor: nothing past its end is read)
__device__ __forceinline__ void cp_async16_part(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 16-byte shared-memory access at a shared-window address
__device__ __forceinline__ Raw<16> lds16(uint32_t addr) {
  Raw<16> r;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
               : "r"(addr));
  return r;
}
__device__ __forceinline__ void sts16(uint32_t addr, const Raw<16>& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.w[0]), "r"(v.w[1]),
               "r"(v.w[2]), "r"(v.w[3])
               : "memory");
}
// an output's column pointer for granule g0
__device__ __forceinline__ char* gp_out(void* p, int64_t g0) { return (char*)p + g0 * 16; }

// Streamed operands of each operation (in ring slot order).
template <int OP, bool GFULL, bool MFULL>
__host__ __device__ constexpr int streamed_operands() {
  return OP == OP_MOD ? (MFULL ? 3 : 1) : OP == OP_RGA ? 2 : (2 + (GFULL ? 1 : 0) + (MFULL ? 2 : 0));
}

// The fast statistic's row sums of a group of RC rows over the warp: the
// rows are first spread over lane groups (a transpose-reduce: each step
// halves the rows a lane carries and exchanges the other half), then each
// group finishes with a butterfly, so RC rows cost about as many shuffles as
// one.  Returns the sum of row (lane >> (5 - log2 RC)) in every lane.
template <int RC>
__device__ __forceinline__ float warp_sum_rows(const float (&v)[RC]) {
  const int lane = threadIdx.x & 31;
  float z;
  if constexpr (RC == 1) {
    z = v[0];
  } else if constexpr (RC == 2) {
    const bool hi = lane & 16;
    const float send = hi ? v[0] : v[1];
    const float keep = hi ? v[1] : v[0];
    z = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 16));
  } else {
    static_assert(RC == 4, "rows per group: 1, 2 or 4");
    const bool b4 = lane & 16, b3 = lane & 8;
    const float s0 = b4 ? v[0] : v[2], s1 = b4 ? v[1] : v[3];
    const float k0 = b4 ? v[2] : v[0], k1 = b4 ? v[3] : v[1];
    const float w0 = __fadd_rn(k0, __shfl_xor_sync(0xFFFFFFFFu, s0, 16));
    const float w1 = __fadd_rn(k1, __shfl_xor_sync(0xFFFFFFFFu, s1, 16));
    z = __fadd_rn(b3 ? w1 : w0, __shfl_xor_sync(0xFFFFFFFFu, b3 ? w0 : w1, 8));
  }
  constexpr int first = RC == 1 ? 16 : RC == 2 ? 8 : 4;
#pragma unroll
  for (int o = first; o > 0; o >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xFFFFFFFFu, z, o));
  return z;
}

// ALLCOLS: every thread owns VPT valid granules (T * VPT * slices == nvec),
// so no column predicate is evaluated.  A group of RC rows that lies wholly
// inside the CTA's rows takes a path without row predicates; only the last
// group of a ragged chunk checks them.
#ifdef DIT_PIPE_MAXNREG  // tuning builds: cap the registers
#define DIT_PIPE_BOUNDS __maxnreg__(DIT_PIPE_MAXNREG)
#else
#define DIT_PIPE_BOUNDS __launch_bounds__(512)
#endif
// Two fp32 values to two OCP E4M3 codes, each rounded to nearest-even and
// saturated to +-448 (NaN stays NaN): the first value in the low byte, so
// the pair is stored in element order.
__device__ __forceinline__ uint32_t e4m3x2(F2 v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(f2_hi(v)), "f"(f2_lo(v)));
  return r;
}
// a granule's P pairs, each scaled by qinv (one fp32 rounding), as E4M3:
// 8 bytes for 16-bit dtypes, 4 for fp32
template <int P>
__device__ __forceinline__ Raw<2 * P> quantise_e4m3(const F2 (&y)[P], F2 qinv) {
  Raw<2 * P> r;
#pragma unroll
  for (int i = 0; i < P / 2; ++i)
    r.w[i] = e4m3x2(f2_mul(y[2 * i], qinv)) | (e4m3x2(f2_mul(y[2 * i + 1], qinv)) << 16);
  return r;
}

// Phased rows: element i of a 16-byte granule (16 / sizeof(T) elements, pair
// i / 2 of the widened granule) belongs to the row when lo <= i < hi.  The
// row's elements of a granule it shares with a neighbouring row are stored
// one by one, so that the neighbour's elements are never written here.
template <class T>
__device__ __forceinline__ void store_part(char* dst, const Raw<16>& r, int lo, int hi) {
  constexpr int ES = (int)sizeof(T);
#pragma unroll
  for (int i = 0; i < 16 / ES; ++i) {
    if (i < lo || i >= hi) continue;
    if constexpr (ES == 4) {
      Raw<4> v;
      v.w[0] = r.w[i];
      st_stream<4>(dst + i * 4, v);
    } else {
      Raw<2> v;
      v.h = (uint16_t)(r.w[i >> 1] >> ((i & 1) * 16));
      st_stream<2>(dst + i * 2, v);
    }
  }
}
// the granule's elements outside [lo, hi) set to zero (they add nothing to
// the row's sum of squares)
template <class T>
__device__ __forceinline__ void mask_part(F2 (&x)[Granule<T>::P], int lo, int hi) {
#pragma unroll
  for (int i = 0; i < Granule<T>::P; ++i) {
    const int e = 2 * i;
    x[i] = f2(e >= lo && e < hi ? f2_lo(x[i]) : 0.0f, e + 1 >= lo && e + 1 < hi ? f2_hi(x[i]) : 0.0f);
  }
}

// The body of one CTA: CTA `cta` of the problem's grid-stride schedule, on
// column slice `slice` of the row.  Q8: the modulated output is OCP E4M3
// (one byte per element, a.out2 for the fused op, a.out otherwise), the
// fp32 value scaled by fl(1 / *a.qscale) first.  PH (phased rows): the row
// pitch is not a multiple of 16 bytes but every streamed tensor starts on a
// 16-byte boundary; one row per group, and the grid is a multiple of the
// period of the rows' offsets modulo 16, so all the rows a CTA takes start
// the same `off` bytes past a 16-byte boundary.  The CTA copies the 16-byte
// granules from that boundary on (a row's first and last granule hold
// elements of its neighbours, masked out of the sum and never stored) and
// holds its [B, 1, D] operands shifted by the same offset.
template <int OP, class T, int VPT, int S, int RC, bool GFULL, bool MFULL, bool ALLCOLS,
          bool Q8 = false, bool PH = false, bool EX = false>
__device__ __forceinline__ void pipe_body(const RowArgs& a, const int64_t cta, const int64_t slice) {
  using G = Granule<T>;
  constexpr int P = G::P;  // fp32 pairs per 16-byte granule
  constexpr int NS = streamed_operands<OP, GFULL, MFULL>();
  constexpr bool kReduce = OP != OP_RGA;
  constexpr bool kGate = OP != OP_MOD;
  constexpr int kX = 0, kU = 1, kG = 2;                      // ring slots
  constexpr int kSc = (OP == OP_MOD) ? 1 : (GFULL ? 3 : 2);  // full scale
  constexpr int kSh = kSc + 1;                               // full shift

  extern __shared__ Raw<16> ring[];  // [S][RC][NS][VPT][T] granules
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = nthr >> 5;

  static_assert(!PH || (RC == 1 && !Q8 && !ALLCOLS), "phased rows: one row per group");
  if (cta >= a.ngroups) return;  // uniform over the CTA
  constexpr int ES = (int)sizeof(T);
  constexpr int EPG = 16 / ES;  // elements per granule
  const int64_t pitch = a.D * (int64_t)ES;
  // phased rows: the byte offset of this CTA's rows past a 16-byte boundary
  // (its first row is row `cta`), and the granules a row spans
  int off = 0;
  if constexpr (PH) off = (int)(((uint64_t)cta * (uint64_t)(pitch & 15)) & 15u);
  const int64_t ngran = PH ? (off + pitch + 15) >> 4 : a.nvec;

  // this thread's granules: t + k * T (+ the column slice of the residual gate)
  const int64_t g0 = slice * nthr * VPT + tid;
  bool cval[VPT];
  // phased rows: granule k's slots [lo, hi) belong to the row, packed as
  // byte k = lo | hi << 4 (one register for every k).  A granule past the row
  // (cval false: never read) gets a meaningless byte; such granules are
  // always the higher k, so what spills out of their byte lands above every
  // valid one.
  [[maybe_unused]] uint32_t bounds = 0;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int64_t gk = g0 + (int64_t)k * nthr;
    cval[k] = ALLCOLS || gk < ngran;
    if constexpr (PH) {
      const int64_t e = (gk * 16 - off) / ES;  // the row element at slot 0
      const uint32_t lo = e < 0 ? (uint32_t)-e : 0u;
      const uint32_t hi = a.D - e < EPG ? (uint32_t)(a.D - e) : (uint32_t)EPG;
      bounds |= (lo | hi << 4) << (8 * k);
    }
  }
  [[maybe_unused]] auto plo = [&](int k) { return (int)((bounds >> (8 * k)) & 15u); };
  [[maybe_unused]] auto phi = [&](int k) { return (int)((bounds >> (8 * k + 4)) & 15u); };
  // a phased granule shared with a neighbouring row
  auto partial = [&](int k) {
    if constexpr (PH)
      return ((bounds >> (8 * k)) & 255u) != (uint32_t)EPG << 4;
    else
      return false;
  };
  // phased rows of the residual gate: the warps that own a row's first or
  // last granule take the masked code path, the others the aligned one (a
  // warp-uniform branch; [1,4097,3077] bf16 L2-flushed 21.1 -> 19.2 us).  The
  // reducing operations test every granule instead: the two copies of their
  // larger passes cost them 9-16% on the same shapes.
  constexpr bool kSplit = PH && !kReduce;
  bool edge_warp = false;
  if constexpr (kSplit) {
    bool mine = false;
#pragma unroll
    for (int k = 0; k < VPT; ++k) mine = mine || (cval[k] && partial(k));
    edge_warp = __any_sync(0xFFFFFFFFu, mine);
  }
  const int64_t kstride = (int64_t)nthr * 16;  // bytes between a thread's granules

  // [B, 1, D] operands of batch bb in fp32: gate; 1 + scale (one rounding); shift
  F2 gv[VPT][P], onev[VPT][P], shv[VPT][P];
  auto load_vectors = [&](int64_t bb) {
    if constexpr (PH) {
      // element by element, at the rows' offset (slots outside the row: 0)
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!cval[k]) continue;
        const int lo = plo(k), hi = phi(k);
        const int64_t e0 = ((g0 + (int64_t)k * nthr) * 16 - off) / ES;  // the row element at slot 0
        const int64_t vb = bb * a.vstride + e0 * ES;
        auto elem = [&](const void* v, int i) {
          float f[1] = {0.0f};
          if (i >= lo && i < hi) Vec<T, ES>::widen(ld_bcast<ES>((const char*)v + vb + i * ES), f);
          return f[0];
        };
#pragma unroll
        for (int i = 0; i < P; ++i) {
          if constexpr (kGate && !GFULL) gv[k][i] = f2(elem(a.g, 2 * i), elem(a.g, 2 * i + 1));
          if constexpr (kReduce && !MFULL) {
            onev[k][i] = f2_add(f2(1.0f, 1.0f), f2(elem(a.sc, 2 * i), elem(a.sc, 2 * i + 1)));
            shv[k][i] = f2(elem(a.sh, 2 * i), elem(a.sh, 2 * i + 1));
          }
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!cval[k]) continue;
        const int64_t vo = bb * a.vstride + g0 * 16 + k * kstride;
        if constexpr (kGate && !GFULL) G::widen(ld_bcast<16>((const char*)a.g + vo), gv[k]);
        if constexpr (kReduce && !MFULL) {
          G::widen(ld_bcast<16>((const char*)a.sc + vo), onev[k]);
#pragma unroll
          for (int i = 0; i < P; ++i) onev[k][i] = f2_add(f2(1.0f, 1.0f), onev[k][i]);
          G::widen(ld_bcast<16>((const char*)a.sh + vo), shv[k]);
        }
      }
    }
  };

  // column pointers (row 0) of the streamed inputs and of the outputs
  const char* gp[NS];
  {
    const void* src[5] = {a.x, a.u, a.g, a.sc, a.sh};
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      int which = i;
      if (OP == OP_MOD && i >= 1) which = 2 + i;              // x, scale, shift
      if (OP == OP_FUSED && !GFULL && i >= 2) which = i + 1;  // h, u, scale, shift
      gp[i] = (const char*)src[which] + g0 * 16;
    }
  }
  char* const out1 = (char*)a.out + g0 * 16;
  // the modulated output: 16 bytes per granule, or 16 / sizeof(T) in E4M3
  constexpr int QB = 16 / (int)sizeof(T);
  char* const out2 = (char*)(OP == OP_FUSED ? a.out2 : a.out) + g0 * (Q8 ? QB : 16);
  const int64_t qpitch = a.D;                   // E4M3 row pitch, bytes
  const int64_t qkstride = (int64_t)nthr * QB;  // bytes between a thread's E4M3 granules
  float qinv_s = 1.0f;
  if constexpr (Q8) qinv_s = __frcp_rn(__ldg(a.qscale));
  const F2 qinv = f2(qinv_s, qinv_s);

  // shared addresses: slot (stage, j, op, k) = stage + j*JS + op*OS + k*KS
  const uint32_t KS = (uint32_t)nthr * 16;
  const uint32_t OS = VPT * KS, JS = NS * OS, SS = RC * JS;
  const uint32_t base = smem_addr(ring) + (uint32_t)tid * 16;
  const uint32_t ring_end = base + S * SS;

  const int64_t nbatch = a.ngroups / a.gpb;  // B
  // group position (batch, group within batch) of the next group to issue
  uint32_t issue_stage = base;
  int64_t ib = cta / a.gpb, ig = cta - ib * a.gpb;
  auto advance = [&](int64_t& bb, int64_t& gg) {
    bb += a.step_b;
    gg += a.step_g;
    if (gg >= a.gpb) {
      gg -= a.gpb;
      ++bb;
    }
  };
  auto issue = [&]() {
    if (ib < nbatch) {
      const int64_t row0 = ib * a.L + ig * RC;
      const int64_t rend = (ib + 1) * a.L;
#pragma unroll
      for (int j = 0; j < RC; ++j) {
        const int64_t row = row0 + j;
        if (row < rend) {
          const int64_t rowoff = row * pitch - off;
          // phased rows: the last row's last granule may run past the
          // tensors' end (uniform test)
          const bool tail = PH && row == a.rows - 1;
#pragma unroll
          for (int op = 0; op < NS; ++op) {
            const char* src = gp[op] + rowoff;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
              if (!cval[k]) continue;
              const uint32_t dst = issue_stage + j * JS + op * OS + k * KS;
              if (tail) {
                const int64_t left = a.rows * pitch - (rowoff + (g0 + (int64_t)k * nthr) * 16);
                if (left < 16) {
                  cp_async16_part(dst, src + k * kstride, (uint32_t)left);
                  continue;
                }
              }
              cp_async16(dst, src + k * kstride);
            }
          }
        }
      }
    }
    cp_async_commit();  // possibly empty: keeps the group count uniform
    advance(ib, ig);
    issue_stage = issue_stage + SS == ring_end ? base : issue_stage + SS;
  };

#pragma unroll
  for (int s = 0; s < S - 1; ++s) issue();
  // the first batch's vectors load while the first groups' copies are in
  // flight (cta < ngroups, so that batch exists)
  int64_t cb = cta / a.gpb, cg = cta - cb * a.gpb;
  int64_t vec_b = cb;  // batch whose vectors are in registers
  load_vectors(cb);

  // per-warp row partials (<= 16 warps); the entries of warps this CTA does
  // not have stay zero (merging a zero pair is exact)
  __shared__ __align__(16) SumPair part[2][RC][16];
  __shared__ uint64_t exact_scratch[16];  // the exact path's warp totals
  __shared__ __align__(16) float partf[2][RC][16];  // the fast statistic's warp sums
  __shared__ float part_scaled[16];                  // and its rescaled sums (rare)
  for (int i = tid; i < 2 * RC * 16; i += nthr)
    if ((i & 15) >= nwarps) {
      (&part[0][0][0])[i] = SumPair{0.0f, 0.0f};
      (&partf[0][0][0])[i] = 0.0f;
    }
  // the statistic's accumulators: two packed slots per thread and row
  constexpr int kNA = 2;
  using Acc = SqAcc<T, kNA>;
  // terms per scalar accumulator: 16-bit P / kNA per granule, fp32 one
  constexpr int kTerms = (sizeof(T) == 2 ? P / kNA : 1) * VPT;
  [[maybe_unused]] const float coef = Acc::coef(kTerms);
  constexpr int kLevels = Log2<Acc::kScalar>::value + 5 + 4;  // thread, warp, 16 warps
  int buf = 0;
  uint32_t stage = base;

  // one group of RC rows starting at row0; CHECK: rows at or past rend are skipped
  auto group = [&](int64_t row0, int64_t rend, auto check_tag) {
    constexpr bool CHECK = decltype(check_tag)::value;
    SumPair ss[RC];
    [[maybe_unused]] float ssf[RC];  // the fast statistic's row sums
    // pass one: the residual (stored), the row sums of squares
    auto pass1 = [&](auto edge_tag) {
      [[maybe_unused]] constexpr bool EDGE = decltype(edge_tag)::value;
#pragma unroll
      for (int j = 0; j < RC; ++j) {
        ss[j] = SumPair{0.0f, 0.0f};
        ssf[j] = 0.0f;
        if (CHECK && row0 + j >= rend) continue;
        [[maybe_unused]] const int64_t rowoff = (row0 + j) * pitch - off;
        Acc acc;
        acc.zero();
        [[maybe_unused]] F2 facc[P];  // fast: independent packed accumulators
#pragma unroll
        for (int i = 0; i < P; ++i) facc[i] = f2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          if (!cval[k]) continue;
          const uint32_t sl = stage + j * JS + k * KS;
          F2 x[P];
          if constexpr (kGate) {
            F2 h[P], u[P], gf[P];
            G::widen(lds16(sl + kX * OS), h);
            G::widen(lds16(sl + kU * OS), u);
            if constexpr (GFULL) G::widen(lds16(sl + kG * OS), gf);
#pragma unroll
            for (int i = 0; i < P; ++i) x[i] = residual_gate2<T>(h[i], u[i], GFULL ? gf[i] : gv[k][i]);
            const Raw<16> r = G::narrow(x);
            if (EDGE && partial(k))
              store_part<T>(out1 + rowoff + k * kstride, r, plo(k), phi(k));
            else
              st_stream<16>(out1 + rowoff + k * kstride, r);
            if constexpr (kReduce) {
              sts16(sl + kX * OS, r);  // the stored residual, read again in pass two
              G::widen(r, x);
            }
          } else {
            G::widen(lds16(sl + kX * OS), x);
          }
          if constexpr (kReduce) {
            if (EDGE && partial(k)) mask_part<T>(x, plo(k), phi(k));
#pragma unroll
            for (int i = 0; i < P; ++i) {
              if constexpr (EX)
                acc.add_pair(i % kNA, x[i]);
              else
                facc[i] = f2_fma(x[i], x[i], facc[i]);
            }
          }
        }
        if constexpr (kReduce) {
          if constexpr (EX)
            ss[j] = acc.total();
          else
          {
#pragma unroll
            for (int i = 1; i < P; ++i) facc[0] = f2_add(facc[0], facc[i]);
            ssf[j] = __fadd_rn(f2_lo(facc[0]), f2_hi(facc[0]));
          }
        }
      }
    };
    if constexpr (!PH) {
      pass1(std::false_type{});
    } else if constexpr (kSplit) {
      if (edge_warp)
        pass1(std::true_type{});
      else
        pass1(std::false_type{});
    } else {
      pass1(std::true_type{});
    }

    if constexpr (kReduce) {
      float rr[RC];
      if constexpr (!EX) {
        // the fast statistic: the RC rows spread over lane groups of the warp,
        // then the warps' sums -- lane l finishes row l % RC with a tree of
        // 16-byte loads and broadcasts it
        const float w = warp_sum_rows<RC>(ssf);
        constexpr int grp_lanes = 32 / RC;
        if ((lane & (grp_lanes - 1)) == 0) partf[buf][lane / grp_lanes][warp] = w;
        __syncthreads();
        const int jr = lane % RC;
        const float4* pp = reinterpret_cast<const float4*>(&partf[buf][jr][0]);
        const float4 p0 = pp[0], p1 = pp[1];
        float tot = __fadd_rn(__fadd_rn(__fadd_rn(p0.x, p0.y), __fadd_rn(p0.z, p0.w)),
                              __fadd_rn(__fadd_rn(p1.x, p1.y), __fadd_rn(p1.z, p1.w)));
        if (nwarps > 8) {  // uniform
          const float4 p2 = pp[2], p3 = pp[3];
          tot = __fadd_rn(tot, __fadd_rn(__fadd_rn(__fadd_rn(p2.x, p2.y), __fadd_rn(p2.z, p2.w)),
                                         __fadd_rn(__fadd_rn(p3.x, p3.y), __fadd_rn(p3.z, p3.w))));
        }
        const float rl = fast_inverse_rms(tot, a.d_f, a.inv_d, a.eps);
#pragma unroll
        for (int j = 0; j < RC; ++j) rr[j] = RC == 1 ? rl : __shfl_sync(0xFFFFFFFFu, rl, j);
        // rare: a row's sum outside the fast range (uniform over the CTA:
        // every warp summed the same partials) -- its squares again, scaled
        if (__any_sync(0xFFFFFFFFu, !fast_sum_in_range(tot))) {
#pragma unroll
          for (int j = 0; j < RC; ++j) {
            const float totj = RC == 1 ? tot : __shfl_sync(0xFFFFFFFFu, tot, j);
            if ((CHECK && row0 + j >= rend) || fast_sum_in_range(totj)) continue;
            const float sc = fast_rescale(totj);
            float s2 = 0.0f;
            const uint32_t sl0 = stage + j * JS + kX * OS;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
              if (!cval[k]) continue;
              F2 x[P];
              G::widen(lds16(sl0 + k * KS), x);
              if constexpr (PH) {
                const uint32_t bk = (bounds >> (8 * k)) & 255u;
                if (bk != (uint32_t)EPG << 4) mask_part<T>(x, (int)(bk & 15u), (int)(bk >> 4));
              }
#pragma unroll
              for (int i = 0; i < P; ++i) {
                const float u0 = __fmul_rn(f2_lo(x[i]), sc), u1 = __fmul_rn(f2_hi(x[i]), sc);
                s2 = __fmaf_rn(u1, u1, __fmaf_rn(u0, u0, s2));
              }
            }
            s2 = warp_sum(s2);
            if (lane == 0) part_scaled[warp] = s2;
            __syncthreads();
            float S2 = 0.0f;
            for (int w = 0; w < nwarps; ++w) S2 = __fadd_rn(S2, part_scaled[w]);
            __syncthreads();  // read before the next row's writes
            rr[j] = fast_inverse_rms_scaled(S2, sc, a.d_f, a.inv_d, a.eps);
          }
        }
      } else {
        // row pairs: merged over the warp, then over the warps (lane l of
        // every warp takes warp l % 16's pair, a 16-lane butterfly merges them)
#pragma unroll
        for (int j = 0; j < RC; ++j) {
          const SumPair w = warp_merge(ss[j]);
          if (lane == 0) part[buf][j][warp] = w;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < RC; ++j) {
          const SumPair p = group_merge<16>(part[buf][j][lane & 15]);
          // the exact path reads the row back from this thread's ring slots
          const uint32_t sl0 = stage + j * JS + kX * OS;
          auto each = [=](auto&& f) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
              if (!cval[k]) continue;
              F2 x[P];
              G::widen(lds16(sl0 + k * KS), x);
              if constexpr (PH) {
                const uint32_t bk = (bounds >> (8 * k)) & 255u;
                if (bk != (uint32_t)EPG << 4) mask_part<T>(x, (int)(bk & 15u), (int)(bk >> 4));
              }
#pragma unroll
              for (int i = 0; i < P; ++i) {
                f(f2_lo(x[i]));
                f(f2_hi(x[i]));
              }
            }
          };
          rr[j] = row_inverse_rms(p, coef, kLevels, a.D, a.d_f, a.eps, each, CtaRow{exact_scratch});
        }
      }
      buf ^= 1;
      // pass two: normalise, modulate, store
      auto pass2 = [&](auto edge_tag) {
        [[maybe_unused]] constexpr bool EDGE = decltype(edge_tag)::value;
#pragma unroll
        for (int j = 0; j < RC; ++j) {
          const float r = rr[j];
          if (CHECK && row0 + j >= rend) continue;
          [[maybe_unused]] const int64_t rowoff = (row0 + j) * pitch - off;
          const F2 r2 = f2(r, r);
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            if (!cval[k]) continue;
            const uint32_t sl = stage + j * JS + k * KS;
            F2 x[P], y[P];
            G::widen(lds16(sl + kX * OS), x);
            if constexpr (MFULL) {
              F2 sc[P], sh[P];
              G::widen(lds16(sl + kSc * OS), sc);
              G::widen(lds16(sl + kSh * OS), sh);
#pragma unroll
              for (int i = 0; i < P; ++i)
                y[i] = modulate2(f2_mul(x[i], r2), f2_add(f2(1.0f, 1.0f), sc[i]), sh[i]);
            } else {
#pragma unroll
              for (int i = 0; i < P; ++i) y[i] = modulate2(f2_mul(x[i], r2), onev[k][i], shv[k][i]);
            }
            if constexpr (Q8)
              st_stream<2 * P>(out2 + (row0 + j) * qpitch + k * qkstride, quantise_e4m3<P>(y, qinv));
            else if (EDGE && partial(k))
              store_part<T>(out2 + rowoff + k * kstride, G::narrow(y), plo(k), phi(k));
            else
              st_stream<16>(out2 + rowoff + k * kstride, G::narrow(y));
          }
        }
      };
      pass2(std::integral_constant<bool, PH>{});
    }
  };

  while (cb < nbatch) {
    cp_async_wait<S - 2>();  // this thread's copies of this group have landed
    issue();                 // refill the stage consumed by the previous group
    if (cb != vec_b) {       // uniform over the CTA
      load_vectors(cb);
      vec_b = cb;
    }
    const int64_t row0 = cb * a.L + cg * RC;
    const int64_t rend = (cb + 1) * a.L;
    if (row0 + RC <= rend)
      group(row0, rend, std::false_type{});
    else
      group(row0, rend, std::true_type{});
    stage = stage + SS == ring_end ? base : stage + SS;
    advance(cb, cg);
  }
  cp_async_wait<0>();  // no copy may outlive the CTA's shared memory
}

template <int OP, class T, int VPT, int S, int RC, bool GFULL, bool MFULL, bool ALLCOLS,
          bool Q8 = false, bool PH = false, bool EX = false>
__global__ void DIT_PIPE_BOUNDS pipe_kernel(RowArgs a) {
  pipe_body<OP, T, VPT, S, RC, GFULL, MFULL, ALLCOLS, Q8, PH, EX>(a, blockIdx.x, blockIdx.y);
}

// The fused op's own entry, held to 80 registers: at its natural 94 two
// 256-thread CTAs fit per SM, at 80 three (same-box, [1,32640,4096] bf16:
// +2% in the hot-path step, the E4M3 variant 0.89 -> 0.98 of copy; 3-6% on
// L2-flushed calls of every shape; no spills).  A register cap on the other
// operations' kernels raised their allocation instead (ptxas uses the cap),
// so they keep the plain launch bound.
#ifndef DIT_PIPE_FUSED_MAXNREG
#define DIT_PIPE_FUSED_MAXNREG 80
#endif
#ifdef DIT_PIPE_MAXNREG
#define DIT_PIPE_FUSED_BOUNDS DIT_PIPE_BOUNDS
#else
#define DIT_PIPE_FUSED_BOUNDS __maxnreg__(DIT_PIPE_FUSED_MAXNREG)  // 80 x 512 threads fit
#endif
template <class T, int VPT, int S, int RC, bool GFULL, bool MFULL, bool ALLCOLS, bool Q8 = false,
          bool PH = false, bool EX = false>
__global__ void DIT_PIPE_FUSED_BOUNDS pipe_fused_kernel(RowArgs a) {
  pipe_body<OP_FUSED, T, VPT, S, RC, GFULL, MFULL, ALLCOLS, Q8, PH, EX>(a, blockIdx.x, blockIdx.y);
}

// The fused op on phased rows: its own entry and register cap.  At 80 it
// spilled; under 104 ptxas takes 94 (no spill; two 224-thread CTAs per SM,
// as ncu shows, against three at 80), the fastest of the caps 80/88/96/104 on
// [1,4097,3077] 16-bit (L2-flushed 38.9 -> 35.7 us; fp32 unchanged).
#ifndef DIT_PIPE_FUSED_PH_MAXNREG
#define DIT_PIPE_FUSED_PH_MAXNREG 104
#endif
#ifdef DIT_PIPE_MAXNREG
#define DIT_PIPE_FUSED_PH_BOUNDS DIT_PIPE_BOUNDS
#else
#define DIT_PIPE_FUSED_PH_BOUNDS __maxnreg__(DIT_PIPE_FUSED_PH_MAXNREG)
#endif
template <class T, int VPT, int S, int RC, bool GFULL, bool MFULL, bool EX>
__global__ void DIT_PIPE_FUSED_PH_BOUNDS pipe_fused_phased_kernel(RowArgs a) {
  pipe_body<OP_FUSED, T, VPT, S, RC, GFULL, MFULL, false, false, true, EX>(a, blockIdx.x, blockIdx.y);
}

// The kernel of one instantiation of the staged row path.
template <int OP, class T, int VPT, int S, int RC, bool GFULL, bool MFULL, bool ALLCOLS, bool Q8,
          bool PH, bool EX>
constexpr auto pipe_kernel_for() {
  if constexpr (OP == OP_FUSED && PH)
    return pipe_fused_phased_kernel<T, VPT, S, RC, GFULL, MFULL, EX>;
  else if constexpr (OP == OP_FUSED)
    return pipe_fused_kernel<T, VPT, S, RC, GFULL, MFULL, ALLCOLS, Q8, false, EX>;
  else
    return pipe_kernel<OP, T, VPT, S, RC, GFULL, MFULL, ALLCOLS, Q8, PH, EX>;
}

// Several problems of one operation in one launch: problem p owns the CTAs
// [begin[p], begin[p+1]), slices[p] per schedule position (column slices of
// the residual gate's long rows; 1 otherwise).  Every problem runs the same
// body with the launch's common block size; threads past a problem's
// narrower row own no granules.  Problem 0 is the largest: its CTAs read
// their arguments as constant-bank operands, exactly as the single-problem
// kernel does (ALLCOLS0: its rows fill every thread's granules); the other
// problems' CTAs first copy their arguments to shared memory, since a kernel
// parameter selected by a runtime index is not a constant-bank operand and
// the body reads some of them for every row group.
struct GroupArgs {
  RowArgs p[kMaxGroup];
  int64_t begin[kMaxGroup + 1];
  int32_t slices[kMaxGroup];
  int32_t count;
};

// Two bodies are inlined; the register bound keeps the modulation at the
// occupancy of its single-problem kernel (<= 64 registers: four 256-thread
// CTAs per SM).  The residual gate's ring (RC rows per stage) and the fused
// op's registers hold them at fewer CTAs per SM anyway.
template <int OP>
constexpr int group_min_blocks() { return OP == OP_MOD ? 2 : 1; }

template <int OP, class T, int VPT, int S, int RC, bool GFULL, bool MFULL, bool ALLCOLS0, bool EX>
__global__ void __launch_bounds__(512, group_min_blocks<OP>())
    pipe_group_kernel(const __grid_constant__ GroupArgs ga) {
  if ((int64_t)blockIdx.x < ga.begin[1]) {  // uniform over the CTA
    const int64_t sl = ga.slices[0];
    const int64_t cta = (int64_t)blockIdx.x / sl;
    pipe_body<OP, T, VPT, S, RC, GFULL, MFULL, ALLCOLS0, false, false, EX>(
        ga.p[0], cta, (int64_t)blockIdx.x - cta * sl);
    return;
  }
  int p = 1;
  while (p + 1 < ga.count && (int64_t)blockIdx.x >= ga.begin[p + 1]) ++p;  // uniform
  const int64_t local = (int64_t)blockIdx.x - ga.begin[p];
  const int64_t sl = ga.slices[p];
  static_assert(sizeof(RowArgs) % 8 == 0, "RowArgs is copied in 8-byte words");
  __shared__ __align__(16) RowArgs sa;
  if (threadIdx.x < sizeof(RowArgs) / 8)
    reinterpret_cast<uint64_t*>(&sa)[threadIdx.x] =
        reinterpret_cast<const uint64_t*>(&ga.p[p])[threadIdx.x];
  __syncthreads();
  const int64_t cta = local / sl;
  pipe_body<OP, T, VPT, S, RC, GFULL, MFULL, false, false, false, EX>(sa, cta, local - cta * sl);
}

// Stages and rows per stage of each operation (tuning builds may override).
#ifndef DIT_PIPE_S_RGA
#define DIT_PIPE_S_RGA 2
#endif
#ifndef DIT_PIPE_RC_RGA
#define DIT_PIPE_RC_RGA 4
#endif
#ifndef DIT_PIPE_S_MOD
#define DIT_PIPE_S_MOD 2
#endif
#ifndef DIT_PIPE_RC_MOD
#define DIT_PIPE_RC_MOD 1
#endif
#ifndef DIT_PIPE_S_FUSED
#define DIT_PIPE_S_FUSED 2
#endif
#ifndef DIT_PIPE_RC_FUSED
#define DIT_PIPE_RC_FUSED 1
#endif
// 16-byte granules per thread per row (tuning builds may override)
#ifndef DIT_PIPE_VPT_RGA
#define DIT_PIPE_VPT_RGA 2
#endif
#ifndef DIT_PIPE_VPT_MOD
#define DIT_PIPE_VPT_MOD 2
#endif
#ifndef DIT_PIPE_VPT_FUSED
#define DIT_PIPE_VPT_FUSED 2
#endif
template <int OP>
__host__ __device__ constexpr int pipe_vpt() {
  return OP == OP_RGA ? DIT_PIPE_VPT_RGA : OP == OP_MOD ? DIT_PIPE_VPT_MOD : DIT_PIPE_VPT_FUSED;
}
constexpr int kPipeBlockMax = 512;    // threads: rows up to 16 KB
constexpr int kStaticSmemReserve = 1024;  // bytes kept for the static arrays

// Let kernel `fn` take more than the default 48 KB of shared memory: once per
// (kernel, device), its dynamic shared memory cap is raised to the most any
// launch here asks for (the opt-in limit less the static reserve), so the cap
// never shrinks under a launch from another host thread.  `opted`: that
// kernel's per-device flags.
constexpr int kOptinDevices = 64;
inline cudaError_t allow_dynamic_smem(const void* fn, const DeviceInfo& dev, size_t smem,
                                      std::atomic<int>* opted) {
  if (smem + kStaticSmemReserve <= 48 * 1024) return cudaSuccess;
  const bool cached = dev.device >= 0 && dev.device < kOptinDevices;
  if (cached && opted[dev.device].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             dev.smem_optin - kStaticSmemReserve);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // do not leave it for the next call to report
    return e;
  }
  if (cached) opted[dev.device].store(1, std::memory_order_release);
  return cudaSuccess;
}

// stages of the phased kernel (one row per stage)
#ifndef DIT_PIPE_S_PHASED
#define DIT_PIPE_S_PHASED 2
#endif
template <int OP>
__host__ __device__ constexpr int pipe_stages() {
  return OP == OP_RGA ? DIT_PIPE_S_RGA : OP == OP_MOD ? DIT_PIPE_S_MOD : DIT_PIPE_S_FUSED;
}
// The E4M3-output modulation moves 3 bytes per element instead of 4, so one
// row per stage leaves too few bytes in flight per CTA: it stages two rows
// (same-box sweep on [1,32640,4096] bf16: 0.76 -> 0.90 of copy), while the
// bf16-output modulation is fastest with one.
#ifndef DIT_PIPE_RC_MOD_Q8
#define DIT_PIPE_RC_MOD_Q8 2
#endif
template <int OP, bool Q8 = false>
__host__ __device__ constexpr int pipe_rows() {
  return OP == OP_RGA ? DIT_PIPE_RC_RGA
                      : OP == OP_MOD ? (Q8 ? DIT_PIPE_RC_MOD_Q8 : DIT_PIPE_RC_MOD) : DIT_PIPE_RC_FUSED;
}

// Launch the staged kernel with S stages; returns cudaErrorNotSupported when
// the row is too long for it (the caller then uses the two-pass kernel).
template <int OP, class T, int S, int RC, bool GFULL, bool MFULL, bool ALLCOLS, bool Q8, bool PH,
          bool EX>
cudaError_t launch_pipe_s(const DeviceInfo& dev, RowArgs a, int64_t B, int block,
                          unsigned slices, size_t smem, cudaStream_t stream) {
  auto kern = pipe_kernel_for<OP, T, pipe_vpt<OP>(), S, RC, GFULL, MFULL, ALLCOLS, Q8, PH, EX>();
  static std::atomic<int> opted[kOptinDevices];
  const cudaError_t e = allow_dynamic_smem((const void*)kern, dev, smem, opted);
  if (e != cudaSuccess) return e;
  // one wave of resident CTAs, each striding over the groups
  a.gpb = (a.L + RC - 1) / RC;
  a.ngroups = B * a.gpb;
  int64_t G = (int64_t)dev.sm_count * resident_ctas(dev, (const void*)kern, block, smem);
  if (G > a.ngroups) G = a.ngroups;
  if constexpr (PH) {
    // rows r and r + G start at the same offset modulo 16 bytes when G is a
    // multiple of 16 / gcd(pitch, 16) (a power of two, at most 8)
    const int64_t m = (a.D * (int64_t)sizeof(T)) & 15;
    const int64_t period = m ? 16 / (m & -m) : 1;
    if (G < a.ngroups) G -= G % period;
  }
  if (G < 1) G = 1;
  if (G > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  a.step_b = G / a.gpb;
  a.step_g = G - a.step_b * a.gpb;
  kern<<<dim3((unsigned)G, slices, 1), dim3((unsigned)block, 1, 1), smem, stream>>>(a);
  return cudaGetLastError();
}

// Depth by shape (same-box sweeps, graph-replayed and L2-flushed, bf16 rows
// of 3072-4608 elements): the residual gate's four rows per stage fill a
// CTA's 128 KB ring, one CTA per SM, which pays off only with many rows per
// SM ([1,32640,4096]); with fewer ([1,8160,4096], [1,4096,4608]) two rows
// per stage and more CTAs are faster (31.5 -> 29.8 and 24.0 -> 19.7 us
// graph-replayed, 31.4 -> 29.3 and 25.2 -> 23.2 us flushed).  The modulation
// goes the other way, from one row per stage to two, below the same bound
// (L2-flushed calls: [1,4096,4608] 23.3 -> 20.8 us, [1,8160,4096] 32.9 ->
// 30.6 us); with many rows per SM one row stays faster inside a stream of
// other kernels (the hot-path step: 6346 vs 6070 GB/s on [1,32640,4096]).
constexpr int64_t kRgaDeepRowsPerSm = 128;  // below: 2 rows per stage

// phased: rows whose pitch is not a multiple of 16 bytes, every streamed
// tensor 16-byte aligned (one row per group; see pipe_body).
template <int OP, bool GFULL, bool MFULL, bool Q8, bool EX>
cudaError_t launch_pipe(const DeviceInfo& dev, int dtype, RowArgs a, int64_t B,
                        cudaStream_t stream, bool phased = false) {
  constexpr int NS = streamed_operands<OP, GFULL, MFULL>();
  constexpr int RC = pipe_rows<OP, Q8>();
  if (Q8 && phased) return cudaErrorNotSupported;
  const int64_t row_bytes = a.D * (dtype == 2 ? 4 : 2);
  // granules per row (phased: at most, over the rows' offsets)
  a.nvec = phased ? (row_bytes + 30) / 16 : row_bytes / 16;
  constexpr int VPT = pipe_vpt<OP>();
  const int64_t threads_needed = (a.nvec + VPT - 1) / VPT;
  const int64_t rows_per_sm = B * a.L / (dev.sm_count > 0 ? dev.sm_count : 1);
  // an RC = 2 variant exists: the residual gate (default 4) and the
  // 16-bit-output modulation (default 1)
  constexpr bool kTwoRowsToo = (OP == OP_RGA && RC > 2) || (OP == OP_MOD && RC == 1);
  const bool two_rows = kTwoRowsToo && rows_per_sm < kRgaDeepRowsPerSm;
  const int rc = phased ? 1 : two_rows ? 2 : RC;
  const size_t limit = (size_t)(dev.smem_optin - kStaticSmemReserve);
  constexpr int SD = pipe_stages<OP>();
  int block;
  unsigned slices = 1;
  if (OP == OP_RGA) {
    // the widest block whose ring fits (at most kPipeBlockMax threads), then
    // equal column slices: a row of 576 granules runs as one 288-thread slice,
    // not as 256 + 32 busy threads of two 256-thread slices
    int64_t bmax = (int64_t)(limit / ((size_t)rc * NS * VPT * 16 * SD)) / 32 * 32;
    if (bmax > kPipeBlockMax) bmax = kPipeBlockMax;
    if (bmax < 32) bmax = 32;
    const int64_t s = (threads_needed + bmax - 1) / bmax;
    if (s > 65535) return cudaErrorInvalidConfiguration;
    slices = (unsigned)s;
    block = (int)(((threads_needed + s - 1) / s + 31) / 32 * 32);
  } else {
    if (threads_needed > kPipeBlockMax) return cudaErrorNotSupported;
    block = (int)((threads_needed + 31) / 32 * 32);
  }
  const size_t per_stage = (size_t)rc * NS * VPT * block * 16;
  int S = SD;
  while (S > 2 && per_stage * S > limit) S = S > 3 ? 3 : 2;  // smaller rings
  if (per_stage * S > limit) return cudaErrorNotSupported;
  const bool allcols = !phased && (int64_t)block * VPT * slices == a.nvec;
  return dispatch_dtype_width(dtype, 16, [&](auto tt, auto) -> cudaError_t {
    using T = typename decltype(tt)::type;
    auto go = [&](auto stages, auto rows, auto cols, auto ph) -> cudaError_t {
      constexpr int SS_ = decltype(stages)::value;
      constexpr int RR_ = decltype(rows)::value;
      return launch_pipe_s<OP, T, SS_, RR_, GFULL, MFULL, decltype(cols)::value, Q8,
                           decltype(ph)::value, EX>(dev, a, B, block, slices, SS_ * per_stage,
                                                    stream);
    };
    auto by_cols = [&](auto stages, auto rows) -> cudaError_t {
      return allcols ? go(stages, rows, std::true_type{}, std::false_type{})
                     : go(stages, rows, std::false_type{}, std::false_type{});
    };
    auto by_rows = [&](auto stages) -> cudaError_t {
      if constexpr (!Q8) {
        if (phased) {
          constexpr int SP = DIT_PIPE_S_PHASED;
          if (SP > 2 && per_stage * SP <= limit)
            return go(std::integral_constant<int, SP>{}, std::integral_constant<int, 1>{},
                      std::false_type{}, std::true_type{});
          return go(std::integral_constant<int, 2>{}, std::integral_constant<int, 1>{},
                    std::false_type{}, std::true_type{});
        }
      }
      if constexpr (kTwoRowsToo)
        if (two_rows) return by_cols(stages, std::integral_constant<int, 2>{});
      return by_cols(stages, std::integral_constant<int, RC>{});
    };
    // instantiated stage counts: the default, 3 and 2 (when the default ring
    // does not fit in shared memory)
    if constexpr (SD == 2) {
      return by_rows(std::integral_constant<int, 2>{});
    } else {
      if (S == SD) return by_rows(std::integral_constant<int, SD>{});
      if constexpr (SD > 3)
        if (S == 3) return by_rows(std::integral_constant<int, 3>{});
      return by_rows(std::integral_constant<int, 2>{});
    }
  });
}

// Several problems of operation OP in one launch of pipe_group_kernel.  Every
// problem must take the staged path (16-byte aligned rows; for the reducing
// operations, rows of at most kPipeBlockMax * VPT granules); returns
// cudaErrorNotSupported otherwise, having launched nothing.  The block is the
// widest problem's; one wave of resident CTAs is split over the problems in
// proportion to their row groups (at least one schedule position each).
template <int OP, bool GFULL, bool MFULL, bool EX>
cudaError_t launch_pipe_grouped(const DeviceInfo& dev, int dtype, const RowArgs* args_in,
                                const int64_t* B_in, int count, cudaStream_t stream) {
  constexpr int NS = streamed_operands<OP, GFULL, MFULL>();
  constexpr int RC = pipe_rows<OP>();
  constexpr int VPT = pipe_vpt<OP>();
  if (count < 1 || count > kMaxGroup) return cudaErrorInvalidValue;
  const int64_t es = dtype == 2 ? 4 : 2;
  // the largest problem (most elements) first; the others keep their order
  RowArgs args[kMaxGroup];
  int64_t B[kMaxGroup];
  int first = 0;
  for (int p = 1; p < count; ++p)
    if (B_in[p] * args_in[p].L * args_in[p].D > B_in[first] * args_in[first].L * args_in[first].D)
      first = p;
  args[0] = args_in[first];
  B[0] = B_in[first];
  for (int p = 0, q = 1; p < count; ++p)
    if (p != first) {
      args[q] = args_in[p];
      B[q++] = B_in[p];
    }
  int block = 32;
  for (int p = 0; p < count; ++p) {
    const int64_t nvec = args[p].D * es / 16;
    const int64_t threads_needed = (nvec + VPT - 1) / VPT;
    int64_t bp = threads_needed;
    if (OP == OP_RGA) {
      if (bp > 256) bp = 256;
    } else if (bp > kPipeBlockMax) {
      return cudaErrorNotSupported;
    }
    bp = (bp + 31) / 32 * 32;
    if (bp > block) block = (int)bp;
  }
  const size_t per_stage = (size_t)RC * NS * VPT * block * 16;
  const size_t limit = (size_t)(dev.smem_optin - kStaticSmemReserve);
  constexpr int SD = pipe_stages<OP>();
  const int S = per_stage * SD <= limit ? SD : 2;
  if (per_stage * S > limit) return cudaErrorNotSupported;
  int64_t sl[kMaxGroup], units[kMaxGroup], total = 0;
  for (int p = 0; p < count; ++p) {
    const int64_t nvec = args[p].D * es / 16;
    sl[p] = OP == OP_RGA ? (nvec + (int64_t)block * VPT - 1) / ((int64_t)block * VPT) : 1;
    units[p] = B[p] * ((args[p].L + RC - 1) / RC) * sl[p];
    total += units[p];
  }
  const bool allcols0 = (int64_t)block * VPT * sl[0] == args[0].D * es / 16;

  return dispatch_dtype_width(dtype, 16, [&](auto tt, auto) -> cudaError_t {
    using T = typename decltype(tt)::type;
    auto go = [&](auto stages, auto cols) -> cudaError_t {
      constexpr int SS_ = decltype(stages)::value;
      auto kern = pipe_group_kernel<OP, T, VPT, SS_, RC, GFULL, MFULL, decltype(cols)::value, EX>;
      const size_t smem = SS_ * per_stage;
      static std::atomic<int> opted[kOptinDevices];
      const cudaError_t e = allow_dynamic_smem((const void*)kern, dev, smem, opted);
      if (e != cudaSuccess) return e;
      const int64_t wave = (int64_t)dev.sm_count * resident_ctas(dev, (const void*)kern, block, smem);
      // Work units: (row group, column slice) pairs.  A CTA streams its
      // groups one after another, about one per memory round trip, so every
      // problem gets CTAs in proportion to its units -- each CTA then takes
      // about the same number of groups, and a small problem (a short audio
      // stream) is not left to a few CTAs that finish last: units * wave /
      // total schedule positions, at least one and at most the problem's
      // groups.  The largest problem gives back what the minimums
      // take, so the grid stays within one wave (a CTA past the wave would
      // start only when another finishes).  The smaller problems round up:
      // their CTAs must not be the last to finish.
      int64_t cps[kMaxGroup], used = 0;
      for (int p = 0; p < count; ++p) {
        const int64_t ng = B[p] * ((args[p].L + RC - 1) / RC);
        const double want = (double)units[p] * (double)wave / (double)total / (double)sl[p];
        int64_t g = p == 0 ? (int64_t)want : (int64_t)ceil(want);
        if (g > ng) g = ng;
        if (g < 1) g = 1;
        cps[p] = g;
        used += g * sl[p];
      }
      if (used > wave) {
        const int64_t give = (used - wave + sl[0] - 1) / sl[0];
        cps[0] = cps[0] > give ? cps[0] - give : 1;
      }
      GroupArgs ga;
      ga.count = count;
      ga.begin[0] = 0;
      for (int p = 0; p < count; ++p) {
        RowArgs a = args[p];
        a.nvec = a.D * es / 16;
        a.gpb = (a.L + RC - 1) / RC;
        a.ngroups = B[p] * a.gpb;
        a.step_b = cps[p] / a.gpb;
        a.step_g = cps[p] - a.step_b * a.gpb;
        ga.p[p] = a;
        ga.slices[p] = (int32_t)sl[p];
        ga.begin[p + 1] = ga.begin[p] + cps[p] * sl[p];
      }
      for (int p = count; p < kMaxGroup; ++p) {
        ga.p[p] = RowArgs{};
        ga.slices[p] = 1;
        ga.begin[p + 1] = ga.begin[count];
      }
      if (ga.begin[count] > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
      kern<<<(unsigned)ga.begin[count], block, smem, stream>>>(ga);
      return cudaGetLastError();
    };
    auto by_cols = [&](auto stages) -> cudaError_t {
      return allcols0 ? go(stages, std::true_type{}) : go(stages, std::false_type{});
    };
    if constexpr (SD == 2) {
      return by_cols(std::integral_constant<int, 2>{});
    } else {
      return S == SD ? by_cols(std::integral_constant<int, SD>{})
                     : by_cols(std::integral_constant<int, 2>{});
    }
  });
}

// Instantiated once each, in k_instances.cu (the residual gate's in
// k_residual_gate.cu, where it is used).
// f(std::bool_constant<EX>{}) with EX the call's row statistic: the exact
// one or the fast one (the residual gate computes none: always false).
template <int OP, class F>
cudaError_t with_statistic(bool exact, F&& f) {
  if constexpr (OP == OP_RGA)
    return f(std::false_type{});
  else
    return exact ? f(std::true_type{}) : f(std::false_type{});
}

#define DIT_PIPE_SIG(o, g, m, q, e)                                                          \
  template cudaError_t launch_pipe<o, g, m, q, e>(const DeviceInfo&, int, RowArgs, int64_t, \
                                                  cudaStream_t, bool)
#define DIT_GROUPED_SIG(o, g, m, e)                                                              \
  template cudaError_t launch_pipe_grouped<o, g, m, e>(const DeviceInfo&, int, const RowArgs*, \
                                                       const int64_t*, int, cudaStream_t)
extern DIT_PIPE_SIG(OP_MOD, false, false, false, false);
extern DIT_PIPE_SIG(OP_MOD, false, true, false, false);
extern DIT_PIPE_SIG(OP_MOD, false, false, true, false);
extern DIT_PIPE_SIG(OP_MOD, false, true, true, false);
extern DIT_PIPE_SIG(OP_FUSED, false, false, false, false);
extern DIT_PIPE_SIG(OP_FUSED, false, true, false, false);
extern DIT_PIPE_SIG(OP_FUSED, true, false, false, false);
extern DIT_PIPE_SIG(OP_FUSED, true, true, false, false);
extern DIT_PIPE_SIG(OP_FUSED, false, false, true, false);
extern DIT_PIPE_SIG(OP_FUSED, false, true, true, false);
extern DIT_PIPE_SIG(OP_FUSED, true, false, true, false);
extern DIT_PIPE_SIG(OP_FUSED, true, true, true, false);
extern DIT_PIPE_SIG(OP_MOD, false, false, false, true);
extern DIT_PIPE_SIG(OP_MOD, false, true, false, true);
extern DIT_PIPE_SIG(OP_MOD, false, false, true, true);
extern DIT_PIPE_SIG(OP_MOD, false, true, true, true);
extern DIT_PIPE_SIG(OP_FUSED, false, false, false, true);
extern DIT_PIPE_SIG(OP_FUSED, false, true, false, true);
extern DIT_PIPE_SIG(OP_FUSED, true, false, false, true);
extern DIT_PIPE_SIG(OP_FUSED, true, true, false, true);
extern DIT_PIPE_SIG(OP_FUSED, false, false, true, true);
extern DIT_PIPE_SIG(OP_FUSED, false, true, true, true);
extern DIT_PIPE_SIG(OP_FUSED, true, false, true, true);
extern DIT_PIPE_SIG(OP_FUSED, true, true, true, true);
extern DIT_GROUPED_SIG(OP_RGA, false, false, false);
extern DIT_GROUPED_SIG(OP_MOD, false, false, false);
extern DIT_GROUPED_SIG(OP_MOD, false, true, false);
extern DIT_GROUPED_SIG(OP_FUSED, false, false, false);
extern DIT_GROUPED_SIG(OP_FUSED, false, true, false);
extern DIT_GROUPED_SIG(OP_FUSED, true, false, false);
extern DIT_GROUPED_SIG(OP_FUSED, true, true, false);
extern DIT_GROUPED_SIG(OP_MOD, false, false, true);
extern DIT_GROUPED_SIG(OP_MOD, false, true, true);
extern DIT_GROUPED_SIG(OP_FUSED, false, false, true);
extern DIT_GROUPED_SIG(OP_FUSED, false, true, true);
extern DIT_GROUPED_SIG(OP_FUSED, true, false, true);
extern DIT_GROUPED_SIG(OP_FUSED, true, true, true);

}  // namespace dit
