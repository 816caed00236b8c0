// dit_stat.cuh -- the row statistic of the RMSNorm-modulation (sm_103a).
//
// Two statistics, chosen per process (dit_set_statistic); each kernel is
// instantiated once for each, so neither carries the other's registers.
//
// The fast statistic (default).  S = the squares summed in fp32 -- one FMA
// per element into one or a few per-thread accumulators, those added in a
// tree, then butterflies over the warp and a sum over the row's warps; the
// long-row kernel merges its per-vector sums as (hi, lo) pairs,
// since a thread there may take thousands of vectors.  ms = S * fl(1/D) with
// one correction from the exact remainder S - q D (an FMA); v = fl(ms + eps);
// r = rsqrtf(v) and one Newton-Raphson step (fast_inverse_rms).  On
// non-negative terms S's relative error is at most (roundings on the longest
// path) * u, u = 2^-24 -- at most 29 u in these kernels -- and r's then at
// most about 17 u: the modulated value is within 2^-18 of max(|t|, |y|) of
// the correctly rounded one, far below a bf16/fp16 ulp unless the final add
// cancels.  The sum's order depends on the kernel, so two kernels (say, for a
// row in an aligned tensor and the same row in a sub-view off a 16-byte
// boundary) may give different last bits.
//
// The exact statistic: ms = RN32(sum x^2 / D), the exact mean of a row's squares rounded once to
// fp32; v = fl(ms + eps); r = RN32(1 / sqrt(v)), the correctly rounded
// inverse root.  Both are single roundings of exact values, so every kernel
// -- whatever order it sums in -- holds the same fp32 r for a row, and the
// modulated outputs, formed from r by the same IEEE operations in the same
// order, are identical bit for bit whichever kernel computes them.
//
// Fast path.  Each thread sums the squares of its elements as pairs
// (hi, lo) with TwoSum (Knuth): hi + lo is the sum of the terms up to the
// rounding errors of the additions into lo.  A 16-bit value's square is exact
// in fp32; for fp32 inputs the product's rounding error, fma(x, x, -x*x),
// joins lo.  A row's pairs are then merged -- TwoSum of the hi parts, the lo
// parts and that error added, the result renormalised with Fast2Sum -- over
// the thread's accumulators, the warp's lanes and, when a CTA spans the row,
// its warps.  The merged pair (H, L) is within
//     E = (c + 3.01 * levels) * u^2 * H + D * 2^-147,    u = 2^-24,
// of the exact sum: c = k(k+1)/2 for k terms per 16-bit accumulator (one
// rounding of lo per term, |lo| <= k u hi), 2k(k+1) for fp32 (two), 3.01 u^2
// per unit of H for each level of merges, and 2^-147 per element for squares
// below fp32's normal range.  RN32((H + L) / D) is decided from the exact
// remainder of q0 = RN(H / D) (an FMA) against the rounding boundaries next
// to q0.  When the exact sum may lie within E of a boundary -- a tie or
// near-tie, about one row in 10^5 for random data -- or the sum is not
// finite, or too large or too small for these steps, the row takes the exact
// path; the decision depends only on (H, L), which every thread of the row
// holds bit for bit, so the branch is uniform.
//
// Window pass.  A normal row the pair cannot decide first sums its squares
// exactly on the top 62 bits of the sum (64-bit integers, one pass) and
// counts the squares with bits below; that settles every row but a tie or a
// near-tie within a few units of 2^-60 of the sum, which the exact path
// takes.
//
// Exact path.  The squares are summed as a big integer: x = M * 2^e with
// M < 2^24, e >= -149, so x^2 = M^2 * 2^(2e) is an integer multiple of 2^-298
// below 2^256.  One pass per base-2^32 digit of the scaled sum, from the
// lowest digit any square reaches to the highest plus a carry digit: each
// thread adds the 32 bits of its squares that fall in the digit, the row's
// threads add their totals (64-bit; no overflow for D <= 2^24) and the carry
// moves up.  The top 64 bits of the sum are divided by D -- the remainder and
// every lower bit make the sticky bit -- and the quotient is rounded to
// nearest even at fp32's last place (2^-149 below 2^-126).
//
// Inverse root.  y = rsqrtf(v) and one Newton-Raphson step, then exact
// integer tests of the rounding boundaries next to y: for y = M * 2^e the
// boundary above y is m = (2M + 1) * 2^(e-1), and 1/sqrt(v) > m iff
// m^2 v < 1, i.e. (2M + 1)^2 * Mv < 2^k for v = Mv * 2^ev -- a comparison of
// 74-bit integers that is never an equality.
#pragma once

#include <stdint.h>

#include "dit_device.cuh"

namespace dit {

// a - b on a pair, one rounding: b * (-1) + a is exact before the rounding
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) { return f2_fma(b, make_float2(-1.0f, -1.0f), a); }

// s + e = a + b exactly (Knuth's TwoSum; every operation rounded to nearest)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
}

// s + e = a + b exactly when |a| >= |b| (Dekker's Fast2Sum)
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// A partial sum of squares h + l with h >= 0 and |l| <= ulp(h) / 2.
struct SumPair {
  float h, l;
};

// (h1 + l1) + (h2 + l2), renormalised; within 3.01 u^2 (h1 + h2) of the
// exact sum of the two pairs.  Commutative bit for bit (TwoSum's error is
// the exact one), so both lanes of a butterfly step get the same pair.
__device__ __forceinline__ SumPair merge(SumPair a, SumPair b) {
  float s, e;
  two_sum(a.h, b.h, s, e);
  const float w = __fadd_rn(__fadd_rn(a.l, b.l), e);
  SumPair r;
  fast_two_sum(s, w, r.h, r.l);
  return r;
}

__device__ __forceinline__ SumPair normalised(float hi, float lo) {
  SumPair r;
  fast_two_sum(hi, lo, r.h, r.l);
  return r;
}

// NS pairs merged as a balanced tree (NS a power of two): log2(NS) levels
template <int NS>
__device__ __forceinline__ SumPair merge_tree(SumPair (&p)[NS]) {
#pragma unroll
  for (int w = NS / 2; w >= 1; w /= 2) {
#pragma unroll
    for (int i = 0; i < w; ++i) p[i] = merge(p[i], p[i + w]);
  }
  return p[0];
}
template <int N>
struct Log2 {
  static constexpr int value = N <= 1 ? 0 : 1 + Log2<N / 2>::value;
};

// ---------------------------------------------------------------------------
// per-thread accumulation
// ---------------------------------------------------------------------------

// Squares of 16-bit values (exact in fp32) in NA packed (hi, lo) pairs (NA a
// power of two).
template <int NA>
struct Sq16 {
  static constexpr int kScalar = 2 * NA;
  F2 hi[NA], lo[NA];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int a = 0; a < NA; ++a) hi[a] = lo[a] = f2(0.0f, 0.0f);
  }
  __device__ __forceinline__ void add(int a, F2 x) {
    const F2 p = f2_mul(x, x);
    const F2 s = f2_add(hi[a], p);
    const F2 bv = f2_sub(s, hi[a]);
    const F2 av = f2_sub(s, bv);
    const F2 e = f2_add(f2_sub(hi[a], av), f2_sub(p, bv));
    hi[a] = s;
    lo[a] = f2_add(lo[a], e);
  }
  // the fast statistic: the square added with one FMA (lo stays zero), and
  // the thread's plain fp32 sum of its accumulators
  __device__ __forceinline__ void add_fast(int a, F2 x) { hi[a] = f2_fma(x, x, hi[a]); }
  __device__ __forceinline__ float fast_total() const {
    F2 h[NA];
#pragma unroll
    for (int a = 0; a < NA; ++a) h[a] = hi[a];
#pragma unroll
    for (int w = NA / 2; w >= 1; w /= 2) {
#pragma unroll
      for (int i = 0; i < w; ++i) h[i] = f2_add(h[i], h[i + w]);
    }
    return __fadd_rn(h[0].x, h[0].y);
  }
  // the thread's pair: its 2 * NA accumulators renormalised and merged, two
  // at a time in the packed halves, then the two halves (log2(2 NA) levels)
  __device__ __forceinline__ SumPair total() const {
    F2 h[NA], l[NA];
#pragma unroll
    for (int a = 0; a < NA; ++a) {
      h[a] = f2_add(hi[a], lo[a]);
      l[a] = f2_sub(lo[a], f2_sub(h[a], hi[a]));
    }
#pragma unroll
    for (int w = NA / 2; w >= 1; w /= 2) {
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const F2 s = f2_add(h[i], h[i + w]);
        const F2 bv = f2_sub(s, h[i]);
        const F2 av = f2_sub(s, bv);
        const F2 e = f2_add(f2_sub(h[i], av), f2_sub(h[i + w], bv));
        const F2 t = f2_add(f2_add(l[i], l[i + w]), e);
        h[i] = f2_add(s, t);
        l[i] = f2_sub(t, f2_sub(h[i], s));
      }
    }
    SumPair a, b;
    a.h = f2_lo(h[0]);
    a.l = f2_lo(l[0]);
    b.h = f2_hi(h[0]);
    b.l = f2_hi(l[0]);
    return merge(a, b);
  }
  // bound coefficient for k terms per accumulator (one rounding of lo each)
  __host__ __device__ static constexpr float coef(int k) { return 0.5f * k * (k + 1); }
};

// Squares of fp32 values in NS scalar (hi, lo) pairs: the product's rounding
// error fma(x, x, -p) joins lo with the sum's (non-contractible intrinsics).
template <int NS>
struct Sq32 {
  static constexpr int kScalar = NS;
  float hi[NS], lo[NS];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int a = 0; a < NS; ++a) hi[a] = lo[a] = 0.0f;
  }
  __device__ __forceinline__ void add(int a, float x) {
    const float p = __fmul_rn(x, x);
    const float pe = __fmaf_rn(x, x, -p);
    float s, e;
    two_sum(hi[a], p, s, e);
    hi[a] = s;
    lo[a] = __fadd_rn(__fadd_rn(lo[a], e), pe);
  }
  __device__ __forceinline__ void add(int a, F2 x) {
    add(a, f2_lo(x));
    add(a + 1, f2_hi(x));
  }
  __device__ __forceinline__ void add_fast(int a, float x) { hi[a] = __fmaf_rn(x, x, hi[a]); }
  __device__ __forceinline__ float fast_total() const {
    float h[NS];
#pragma unroll
    for (int a = 0; a < NS; ++a) h[a] = hi[a];
#pragma unroll
    for (int w = NS / 2; w >= 1; w /= 2) {
#pragma unroll
      for (int i = 0; i < w; ++i) h[i] = __fadd_rn(h[i], h[i + w]);
    }
    return h[0];
  }
  __device__ __forceinline__ void add_fast(int a, F2 x) {
    add_fast(a, f2_lo(x));
    add_fast(a + 1, f2_hi(x));
  }
  __device__ __forceinline__ SumPair total() const {
    SumPair p[NS];
#pragma unroll
    for (int a = 0; a < NS; ++a) p[a] = normalised(hi[a], lo[a]);
    return merge_tree<NS>(p);
  }
  __host__ __device__ static constexpr float coef(int k) { return 2.0f * k * (k + 1); }
};

// The per-thread accumulator of storage type T with NA packed slots: 16-bit
// types one packed (hi, lo) pair per slot, fp32 two scalar pairs per slot.
template <class T, int NA>
struct SqAcc : Sq16<NA> {
  __device__ __forceinline__ void add_pair(int a, F2 x) { Sq16<NA>::add(a, x); }
  __device__ __forceinline__ void add_pair_fast(int a, F2 x) { Sq16<NA>::add_fast(a, x); }
};
template <int NA>
struct SqAcc<float, NA> : Sq32<2 * NA> {
  __device__ __forceinline__ void add_pair(int a, F2 x) { Sq32<2 * NA>::add(2 * a, x); }
  __device__ __forceinline__ void add_pair_fast(int a, F2 x) { Sq32<2 * NA>::add_fast(2 * a, x); }
};

// ---------------------------------------------------------------------------
// warp-level merge
// ---------------------------------------------------------------------------

// A value summed over the warp (xor butterfly: every lane gets the same sum).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// A value summed over groups of W lanes (xor butterfly; every lane of a
// group gets the same sum: IEEE addition is commutative).
template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// The pair of every lane merged over the warp (5 levels); all lanes return
// the same pair.
__device__ __forceinline__ SumPair warp_merge(SumPair p) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    SumPair q;
    q.h = __shfl_xor_sync(0xFFFFFFFFu, p.h, o);
    q.l = __shfl_xor_sync(0xFFFFFFFFu, p.l, o);
    p = merge(p, q);
  }
  return p;
}
// The same over aligned groups of W lanes (W a power of two <= 32).
template <int W>
__device__ __forceinline__ SumPair group_merge(SumPair p) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) {
    SumPair q;
    q.h = __shfl_xor_sync(0xFFFFFFFFu, p.h, o);
    q.l = __shfl_xor_sync(0xFFFFFFFFu, p.l, o);
    p = merge(p, q);
  }
  return p;
}

// ---------------------------------------------------------------------------
// the rounding of the mean
// ---------------------------------------------------------------------------

// E: the bound on |exact sum - (H + L)| for the merged pair of a row of D
// elements, given the accumulators' coefficient and the merge levels.
__device__ __forceinline__ float sum_bound(float H, float coef, int levels, float Df) {
  const float c = (coef + 3.01f * (float)levels) * 0x1p-48f * 1.0001f;
  return __fmaf_ru(c, H, __fmul_ru(Df, 0x1p-147f));
}

// ms = RN32(S / D) for S within E of H + L (H >= 0, |L| <= ulp(H)/2).
// Returns false, leaving ms unset, when that cannot be decided here.
__device__ __forceinline__ bool mean_from_pair(float H, float L, float E, float Df, float& ms) {
  if (H == 0.0f) {
    // every square rounded to zero in fp32, so each was at most 2^-150 and
    // S / D <= 2^-150, which rounds to zero (2^-150 itself: ties to even)
    ms = 0.0f;
    return true;
  }
  if (!(H < 0x1p120f) || H < __fmul_rn(Df, 0x1p-100f)) return false;  // also NaN
  if (!(fabsf(L) < 0x1p120f)) return false;
  const float q0 = __fdiv_rn(H, Df);
  const float rho = __fmaf_rn(-q0, Df, H);  // H - q0 D, exactly
  const uint32_t qb = __float_as_uint(q0);
  const float nx = __uint_as_float(qb + 1), pv = __uint_as_float(qb - 1);
  const float up = __fsub_rn(nx, q0), dn = __fsub_rn(q0, pv);  // exact spacings
  const float hu = __fmul_rn(__fmul_rn(0.5f, Df), up);          // exact: D < 2^24
  const float hd = __fmul_rn(__fmul_rn(0.5f, Df), dn);
  // S - D * (boundary): computed with two roundings, so within
  // 2u (|rho| + hu + |L|) of its value, plus E
  const float mag = __fadd_ru(__fadd_ru(fabsf(rho), fmaxf(hu, hd)), fabsf(L));
  const float marg = __fmaf_ru(0x1p-22f, mag, E);
  const float d_up = __fadd_rn(__fsub_rn(rho, hu), L);
  const float d_dn = __fadd_rn(__fadd_rn(rho, hd), L);
  if (d_up < -marg && d_dn > marg) {
    ms = q0;
    return true;
  }
  if (d_up > marg) {  // above q0's upper boundary: below nx's upper one?
    const float up2 = __fsub_rn(__uint_as_float(qb + 2), nx);
    const float hu2 = __fmul_rn(__fmul_rn(0.5f, Df), up2);
    const float d2 = __fadd_rn(__fsub_rn(__fsub_rn(rho, __fmul_rn(2.0f, hu)), hu2), L);
    const float mag2 = __fadd_ru(__fadd_ru(mag, __fmul_ru(2.0f, hu)), hu2);
    if (d2 < -__fmaf_ru(0x1p-21f, mag2, E)) {
      ms = nx;
      return true;
    }
    return false;
  }
  if (d_dn < -marg) {  // below q0's lower boundary: above pv's lower one?
    const float dn2 = __fsub_rn(pv, __uint_as_float(qb - 2));
    const float hd2 = __fmul_rn(__fmul_rn(0.5f, Df), dn2);
    const float d2 = __fadd_rn(__fadd_rn(__fadd_rn(rho, __fmul_rn(2.0f, hd)), hd2), L);
    const float mag2 = __fadd_ru(__fadd_ru(mag, __fmul_ru(2.0f, hd)), hd2);
    if (d2 > __fmaf_ru(0x1p-21f, mag2, E)) {
      ms = pv;
      return true;
    }
    return false;
  }
  return false;
}

// Combiners over the threads that hold a row, for the exact path.  Every
// thread of the row calls each member the same number of times.
struct WarpRow {
  __device__ __forceinline__ uint64_t sum(uint64_t v) const {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
  }
  __device__ __forceinline__ int imin(int v) const {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
  }
  __device__ __forceinline__ int imax(int v) const {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
  }
  __device__ __forceinline__ bool any(bool b) const { return __any_sync(0xFFFFFFFFu, b); }
};

// A CTA spanning the row: warp totals through `scratch` (one 64-bit word per
// warp), two barriers per call; every thread combines the words in the same
// order.  (min / max take values >= -1: they are offset by one into
// unsigned order.)
struct CtaRow {
  uint64_t* scratch;
  __device__ __forceinline__ uint64_t sum(uint64_t v) const {
    return combine(WarpRow().sum(v), 0u, [](uint64_t a, uint64_t b) { return a + b; });
  }
  __device__ __forceinline__ int imin(int v) const {
    const uint64_t u = (uint64_t)(int64_t)(WarpRow().imin(v) + 1);
    return (int)combine(u, ~0ull, [](uint64_t a, uint64_t b) { return a < b ? a : b; }) - 1;
  }
  __device__ __forceinline__ int imax(int v) const {
    const uint64_t u = (uint64_t)(int64_t)(WarpRow().imax(v) + 1);
    return (int)combine(u, 0u, [](uint64_t a, uint64_t b) { return a > b ? a : b; }) - 1;
  }
  __device__ __forceinline__ bool any(bool b) const { return __syncthreads_or(b) != 0; }

 private:
  template <class Op>
  __device__ __forceinline__ uint64_t combine(uint64_t v, uint64_t init, Op op) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    uint64_t t = init;
    for (int w = 0; w < nw; ++w) t = op(t, scratch[w]);
    __syncthreads();
    return t;
  }
};

// x = M * 2^e (M < 2^24, e >= -149) from |x|'s fp32 bits (finite, nonzero);
// returns the bit of the 2^-298-scaled sum where M^2 starts.
__device__ __forceinline__ int square_position(uint32_t b, uint64_t& M) {
  const uint32_t E = b >> 23;
  M = E ? (uint64_t)((b & 0x7FFFFFu) | 0x800000u) : (uint64_t)b;
  return 2 * ((int)(E ? E : 1u) - 150) + 298;
}

// The 32 bits of x^2 (scaled by 2^298) in digit j of the sum.
__device__ __forceinline__ uint32_t square_digit(float x, int j) {
  const uint32_t b = __float_as_uint(x) & 0x7FFFFFFFu;
  if (b == 0u) return 0u;
  uint64_t M;
  const int sh = square_position(b, M) - 32 * j;
  const uint64_t Q = M * M;  // < 2^48
  if (sh >= 0) return sh < 32 ? (uint32_t)(Q << sh) : 0u;
  return sh > -48 ? (uint32_t)(Q >> -sh) : 0u;
}

// RN32((T + s) * 2^w / D) for a nonzero 64-bit T, where s is 0 or, when
// `sticky`, a positive amount below one unit of T's last bit (1 <= D <= 2^24).
// T is shifted up to bit 63; the quotient by D then keeps at least 40 bits,
// and its bits below fp32's last place, the remainder and `sticky` decide the
// rounding to nearest even (last place 2^-149 below 2^-126; +inf past
// FLT_MAX).
__device__ __forceinline__ float round_quotient(uint64_t T, int w, uint64_t D, bool sticky) {
  const int lz = __clzll((long long)T);
  T <<= lz;
  w -= lz;
  const uint64_t q = T / D;
  sticky = sticky || (T - q * D) != 0u;
  const int top = 63 - __clzll((long long)q);  // q >= 2^63 / 2^24
  int lsb = top - 23;
  if (lsb + w < -149) lsb = -149 - w;  // subnormal result: last place 2^-149
  uint64_t mant = lsb < 64 ? q >> lsb : 0u;
  const int g = lsb - 1;
  const bool guard = g < 64 ? ((q >> g) & 1u) != 0u : false;
  if (g < 64) {
    sticky = sticky || (q & ((1ull << g) - 1u)) != 0u;
  } else {
    sticky = sticky || q != 0u;
  }
  if (guard && (sticky || (mant & 1u))) ++mant;
  // mant * 2^(lsb + w), mant <= 2^24: build the fp32 bits
  if (mant == 0u) return 0.0f;
  int ex = lsb + w;  // exponent of mant's last bit
  if (mant == (1ull << 24)) {
    mant >>= 1;
    ++ex;
  }
  if (mant < (1ull << 23)) return __uint_as_float((uint32_t)mant);  // subnormal (ex == -149)
  const int field = ex + 23 + 127;
  if (field >= 255) return __uint_as_float(0x7F800000u);
  return __uint_as_float(((uint32_t)field << 23) | ((uint32_t)mant & 0x7FFFFFu));
}

// The fp32 value's 2M+1 midpoint above it, times D, in units of 2^lsbe: an
// exact 64-bit integer when it fits (positive normal value given by bits).
__device__ __forceinline__ uint64_t midpoint_times_d(uint32_t qb, uint64_t D, int lsbe) {
  const uint64_t M = (qb & 0x7FFFFFu) | 0x800000u;
  const int e = (int)(qb >> 23) - 150;  // q = M * 2^e; midpoint (2M+1) 2^(e-1)
  return ((2 * M + 1) * D) << (e - 1 - lsbe);
}

// The second tier, for normal rows the pair could not decide: every square
// summed exactly on a window of the sum's top bits.  With 2^eh <= H (H within
// a hair of the sum S, so S < 2^(eh+2)), the window's last bit is
// l = 2^(eh-60): A = sum of floor(x^2 / l) is exact in 64 bits (A <= S / l <
// 2^62), and nb counts the squares with bits below l, so S / l lies in
// [A, A + nb) -- exactly A when nb = 0, strictly inside otherwise.  The mean
// is decided when no rounding boundary of RN32(S / D) lies in [A, A + nb]
// (boundaries m * D / l are exact integers for D <= 2^24).  Returns false when
// one does (a tie or a near-tie closer than nb units of 2^(eh-60)).
template <class Each, class Row>
__device__ __forceinline__ bool window_mean_square(Each each, Row row, float H, int64_t D, float& ms) {
  const int eh = (int)(__float_as_uint(H) >> 23) - 127;
  const int base = eh - 60 + 298;  // the window's last bit, as a bit of the 2^-298-scaled sum
  uint64_t A = 0;
  unsigned nb = 0;
  each([&](float x) {  // no branches: zero gives M = 0
    uint64_t M;
    const int sh = square_position(__float_as_uint(x) & 0x7FFFFFFFu, M) - base;
    const uint64_t Q = M * M;  // < 2^48; Q << sh < 2^62 since x^2 <= S
    const int up = sh > 0 ? sh : 0, down = sh < 0 ? min(-sh, 63) : 0;
    const uint64_t part = (Q >> down) << up;
    A += part;
    nb += ((part >> up) << down) != Q;  // bits below the window
  });
  A = row.sum(A);
  nb = (unsigned)row.sum((uint64_t)nb);
  if (A == 0u) return false;
  const int lsbe = eh - 60;
  const float q = round_quotient(A, lsbe, (uint64_t)D, nb != 0u);
  if (nb == 0u) {  // S = A * 2^lsbe exactly
    ms = q;
    return true;
  }
  const uint32_t qb = __float_as_uint(q);
  if (!(q >= 0x1p-100f) || qb >= 0x7F000000u) return false;
  const uint64_t up = midpoint_times_d(qb, (uint64_t)D, lsbe);
  const uint64_t dn = midpoint_times_d(qb - 1, (uint64_t)D, lsbe);
  if (dn < A && A + nb < up) {
    ms = q;
    return true;
  }
  return false;
}

// Exact RN32(sum x^2 / D) over the row.  `each(f)` calls f(float x) for every
// element of the row that this thread holds; `row` combines over the row's
// threads (WarpRow or CtaRow).
template <class Each, class Row>
__device__ __forceinline__ float exact_mean_square(Each each, Row row, int64_t D) {
  bool nan = false, inf = false;
  int lo = 0x7FFFFFFF, hi = -1;
  each([&](float x) {
    const uint32_t b = __float_as_uint(x) & 0x7FFFFFFFu;
    if (b > 0x7F800000u) {
      nan = true;
    } else if (b == 0x7F800000u) {
      inf = true;
    } else if (b != 0u) {
      uint64_t M;
      const int p = square_position(b, M);
      lo = min(lo, p);
      hi = max(hi, p);
    }
  });
  nan = row.any(nan);
  inf = row.any(inf);
  if (nan) return __uint_as_float(0x7FFFFFFFu);
  if (inf) return __uint_as_float(0x7F800000u);
  lo = row.imin(lo);
  hi = row.imax(hi);
  if (hi < 0) return 0.0f;  // every element is zero
  // digits j0..j1: the squares span bits [lo, hi + 48); the sum of D <= 2^24
  // of them stays below 2^(hi + 72), within one more digit
  const int j0 = lo >> 5, j1 = ((hi + 47) >> 5) + 1;
  uint32_t digit[20];
  uint64_t carry = 0;
  for (int j = j0; j <= j1; ++j) {
    uint64_t part = 0;
    each([&](float x) { part += square_digit(x, j); });
    const uint64_t t = row.sum(part) + carry;
    digit[j - j0] = (uint32_t)t;
    carry = t >> 32;
  }
  // the top 64 bits of the sum, and whether anything lies below them
  int it = j1 - j0;
  while (it > 0 && digit[it] == 0u) --it;
  const uint32_t w2 = digit[it], w1 = it >= 1 ? digit[it - 1] : 0u, w0 = it >= 2 ? digit[it - 2] : 0u;
  bool sticky = false;
  for (int i = 0; i + 2 < it; ++i) sticky = sticky || digit[i] != 0u;
  const int lz = __clz(w2);
  uint64_t T = ((uint64_t)w2 << 32) | w1;
  if (lz > 0) {
    T = (T << lz) | (w0 >> (32 - lz));
    sticky = sticky || (uint32_t)(w0 << lz) != 0u;
  } else {
    sticky = sticky || w0 != 0u;
  }
  // bit 0 of T weighs 2^(32 (it + j0) - 32 - lz - 298)
  return round_quotient(T, 32 * (it + j0) - 32 - lz - 298, (uint64_t)D, sticky);
}

// ---------------------------------------------------------------------------
// the correctly rounded inverse root
// ---------------------------------------------------------------------------

// Whether 1/sqrt(v) lies above the midpoint between the fp32 value y and the
// next one up (y, v positive normal, given by their bits).
__device__ __forceinline__ bool root_above_midpoint(uint32_t yb, uint32_t vb) {
  const uint64_t My = (yb & 0x7FFFFFu) | 0x800000u;
  const int ey = (int)(yb >> 23) - 150;
  const uint64_t Mv = (vb & 0x7FFFFFu) | 0x800000u;
  const int ev = (int)(vb >> 23) - 150;
  const uint64_t P = (2 * My + 1) * (2 * My + 1);  // < 2^50
  const uint64_t zl = P * Mv, zh = __umul64hi(P, Mv);
  const int k = -(2 * ey - 2 + ev);  // above  <=>  P * Mv < 2^k
  if (k >= 128) return true;
  if (k < 0) return false;
  if (k >= 64) return zh < (1ull << (k - 64));
  return zh == 0u && zl < (1ull << k);
}

__device__ __forceinline__ float rsqrt_rn(float v) {
  if (!(v > 0.0f)) return v == 0.0f ? __uint_as_float(0x7F800000u) : v;  // +inf; NaN
  if (v == __uint_as_float(0x7F800000u)) return 0.0f;
  float back = 1.0f;
  if (v < 0x1p-126f) {  // subnormal: 1/sqrt(v 2^64) = 2^-32 / sqrt(v), exactly
    v = __fmul_rn(v, 0x1p64f);
    back = 0x1p32f;
  }
  float y = rsqrtf(v);
  const float e = __fmaf_rn(__fmul_rn(-v, y), y, 1.0f);
  y = __fmaf_rn(__fmul_rn(0.5f, y), e, y);
  uint32_t yb = __float_as_uint(y);
  const uint32_t vb = __float_as_uint(v);
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    if (root_above_midpoint(yb, vb)) {
      ++yb;
    } else if (!root_above_midpoint(yb - 1, vb)) {
      --yb;
    } else {
      break;
    }
  }
  return __fmul_rn(__uint_as_float(yb), back);
}

// The fast statistic (the library's default): from the row's fp32 sum of
// squares S -- each thread's squares added with one FMA each, merged in tree
// order -- ms = S * fl(1/D) with one correction by the exact residual
// S - q D (an FMA; the correctly rounded S / D except in rare near-halfway
// cases), v = fl(ms + eps), and r = rsqrtf(v) refined by one Newton-Raphson
// step.  For S in [2^-100, 2^100] (fast_sum_in_range).
__device__ __forceinline__ float fast_inverse_rms(float S, float Df, float inv_d, float eps) {
  const float q = __fmul_rn(S, inv_d);
  const float ms = __fmaf_rn(__fmaf_rn(-q, Df, S), inv_d, q);
  const float v = __fadd_rn(ms, eps);
  const float y0 = rsqrtf(v);
  const float e = __fmaf_rn(__fmul_rn(-v, y0), y0, 1.0f);
  return __fmaf_rn(__fmul_rn(0.5f, y0), e, y0);
}

// Outside [2^-100, 2^100] the fp32 sum is not a usable statistic: a square
// overflowed (S = +inf, though the row's mean may be finite: one element of
// 3e19), the row holds infinities, or its squares fell below fp32's normal
// range.  The kernels then sum the row's squares again, of x * fast_rescale(S)
// (2^-64 for a large S, 2^64 for a small one), and take r from
// fast_inverse_rms_scaled.  NaN counts as in range: it propagates, as in the
// definition.  The branch is uniform over a row's threads, which hold the
// same S.
__device__ __forceinline__ bool fast_sum_in_range(float S) {
  return !(S < 0x1p-100f) && !(S > 0x1p100f);
}
__device__ __forceinline__ float fast_rescale(float S) { return S > 1.0f ? 0x1p-64f : 0x1p64f; }

// 1 / sqrt(v) for any v >= 0 (rsqrtf and one Newton step on v scaled by an
// even power of two into rsqrtf's range): +0 -> +inf, +inf -> 0, NaN -> NaN.
__device__ __forceinline__ float fast_rsqrt(float v) {
  float w = v, back = 1.0f;
  if (v < 0x1p-100f) {
    w = __fmul_rn(v, 0x1p100f);
    back = 0x1p50f;
  } else if (v > 0x1p100f) {
    w = __fmul_rn(v, 0x1p-100f);
    back = 0x1p-50f;
  }
  if (w == 0.0f) return __int_as_float(0x7f800000);
  if (w == __int_as_float(0x7f800000)) return 0.0f;
  const float y0 = rsqrtf(w);
  const float e = __fmaf_rn(__fmul_rn(-w, y0), y0, 1.0f);
  return __fmul_rn(__fmaf_rn(__fmul_rn(0.5f, y0), e, y0), back);
}

// r from S2, the row's sum of (x * scale)^2 (scale from fast_rescale): the
// mean of the scaled squares, scaled back by 1 / scale^2 = 2^(+-128) in two
// exact steps of 2^64 (the second may overflow to +inf -- then r = 0, as
// when the exact mean rounds past fp32's range -- or round into the
// subnormal range), then v = fl(ms + eps) and r = 1 / sqrt(v).  S2 = +inf
// (an infinity in the row) gives r = 0, NaN gives NaN.
__device__ __forceinline__ float fast_inverse_rms_scaled(float S2, float scale, float Df,
                                                         float inv_d, float eps) {
  // an infinity in the row: ms = +inf, r = 0 (the remainder step would
  // turn inf - inf into NaN)
  if (S2 == __int_as_float(0x7f800000)) return 0.0f;
  const float q = __fmul_rn(S2, inv_d);
  const float mss = __fmaf_rn(__fmaf_rn(-q, Df, S2), inv_d, q);
  const float step = scale < 1.0f ? 0x1p64f : 0x1p-64f;
  const float ms = __fmul_rn(__fmul_rn(mss, step), step);
  return fast_rsqrt(__fadd_rn(ms, eps));
}

// `each` is taken by value (and should capture by value): only the exact
// path, a separate function, needs the row's elements in memory.
template <class Each, class Row>
// r of one row from its merged pair: the fast decision, else the exact path.
// Uniform over the row's threads (they hold the same pair).
__device__ __forceinline__ float row_inverse_rms(SumPair p, float coef, int levels, int64_t D,
                                                 float Df, float eps, const Each& each, Row row) {
  float ms;
  if (!mean_from_pair(p.h, p.l, sum_bound(p.h, coef, levels, Df), Df, ms)) {
    // normal rows: the window pass; ties, and rows the pair cannot stand
    // for (not finite, too large or small), the exact path
    const bool normal = p.h >= __fmul_rn(Df, 0x1p-100f) && p.h < 0x1p120f;
    if (!(normal && window_mean_square(each, row, p.h, D, ms))) ms = exact_mean_square(each, row, D);
  }
  return rsqrt_rn(__fadd_rn(ms, eps));
}

}  // namespace dit
