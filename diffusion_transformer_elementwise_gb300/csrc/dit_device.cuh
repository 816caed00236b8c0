// dit_device.cuh -- device helpers for the DiT elementwise kernels (sm_103a).
//
// * Raw<VB>: VB bytes of storage held in registers (VB = 32, 16, 8, 4 or 2).
// * ld_stream / st_stream: vector accesses for data touched once (activations),
//   issued as one ld/st of VB bytes; 32-byte accesses use the 256-bit vector
//   forms that sm_100-class GPUs add to ld/st.  Loads skip L1 allocation.
// * ld_bcast: vector loads of the small [B, 1, D] operands, which every CTA of
//   a batch re-reads; they go through the read-only path and stay cached.
// * Vec<T, VB>: exact widening of VB bytes of T to fp32 and one
//   round-to-nearest-even narrowing back (cvt.rn; subnormals kept, no FTZ).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dit {

template <int VB>
struct Raw {
  uint32_t w[VB / 4];
};
template <>
struct Raw<2> {
  uint16_t h;
};

// ---------------------------------------------------------------------------
// loads and stores
// ---------------------------------------------------------------------------

template <int VB>
__device__ __forceinline__ Raw<VB> ld_stream(const void* p);
template <int VB>
__device__ __forceinline__ Raw<VB> ld_bcast(const void* p);
template <int VB>
__device__ __forceinline__ void st_stream(void* p, const Raw<VB>& v);

template <>
__device__ __forceinline__ Raw<32> ld_stream<32>(const void* p) {
  Raw<32> r;
  asm volatile(
      "ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
        "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
      : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<16> ld_stream<16>(const void* p) {
  Raw<16> r;
  asm volatile("ld.global.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
               : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<8> ld_stream<8>(const void* p) {
  Raw<8> r;
  asm volatile("ld.global.L1::no_allocate.v2.b32 {%0,%1}, [%2];"
               : "=r"(r.w[0]), "=r"(r.w[1])
               : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<4> ld_stream<4>(const void* p) {
  Raw<4> r;
  asm volatile("ld.global.L1::no_allocate.b32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<2> ld_stream<2>(const void* p) {
  Raw<2> r;
  asm volatile("ld.global.L1::no_allocate.b16 %0, [%1];" : "=h"(r.h) : "l"(p));
  return r;
}

template <>
__device__ __forceinline__ Raw<32> ld_bcast<32>(const void* p) {
  Raw<32> r;
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]),
                 "=r"(r.w[4]), "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<16> ld_bcast<16>(const void* p) {
  Raw<16> r;
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
               : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<8> ld_bcast<8>(const void* p) {
  Raw<8> r;
  asm volatile("ld.global.nc.v2.b32 {%0,%1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<4> ld_bcast<4>(const void* p) {
  Raw<4> r;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(r.w[0]) : "l"(p));
  return r;
}
template <>
__device__ __forceinline__ Raw<2> ld_bcast<2>(const void* p) {
  Raw<2> r;
  asm volatile("ld.global.nc.b16 %0, [%1];" : "=h"(r.h) : "l"(p));
  return r;
}

template <>
__device__ __forceinline__ void st_stream<32>(void* p, const Raw<32>& v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
               "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]),
               "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
               : "memory");
}
template <>
__device__ __forceinline__ void st_stream<16>(void* p, const Raw<16>& v) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
               : "memory");
}
template <>
__device__ __forceinline__ void st_stream<8>(void* p, const Raw<8>& v) {
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1])
               : "memory");
}
template <>
__device__ __forceinline__ void st_stream<4>(void* p, const Raw<4>& v) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(v.w[0]) : "memory");
}
template <>
__device__ __forceinline__ void st_stream<2>(void* p, const Raw<2>& v) {
  asm volatile("st.global.b16 [%0], %1;" ::"l"(p), "h"(v.h) : "memory");
}

// ---------------------------------------------------------------------------
// dtype conversion
// ---------------------------------------------------------------------------

template <class T, int VB>
struct Vec;

// bf16: a 32-bit word holds two elements, the lower address in the low half.
template <int VB>
struct Vec<__nv_bfloat16, VB> {
  static constexpr int N = VB / 2;
  __device__ __forceinline__ static void widen(const Raw<VB>& r, float (&f)[N]) {
#pragma unroll
    for (int i = 0; i < VB / 4; ++i) {
      f[2 * i] = __uint_as_float(r.w[i] << 16);
      f[2 * i + 1] = __uint_as_float(r.w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static Raw<VB> narrow(const float (&f)[N]) {
    Raw<VB> r;
#pragma unroll
    for (int i = 0; i < VB / 4; ++i) {
      __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      r.w[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    return r;
  }
};
template <>
struct Vec<__nv_bfloat16, 2> {
  static constexpr int N = 1;
  __device__ __forceinline__ static void widen(const Raw<2>& r, float (&f)[1]) {
    f[0] = __uint_as_float(static_cast<uint32_t>(r.h) << 16);
  }
  __device__ __forceinline__ static Raw<2> narrow(const float (&f)[1]) {
    Raw<2> r;
    r.h = __bfloat16_as_ushort(__float2bfloat16_rn(f[0]));
    return r;
  }
};

template <int VB>
struct Vec<__half, VB> {
  static constexpr int N = VB / 2;
  __device__ __forceinline__ static void widen(const Raw<VB>& r, float (&f)[N]) {
#pragma unroll
    for (int i = 0; i < VB / 4; ++i) {
      uint32_t w = r.w[i];
      float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w));
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
  __device__ __forceinline__ static Raw<VB> narrow(const float (&f)[N]) {
    Raw<VB> r;
#pragma unroll
    for (int i = 0; i < VB / 4; ++i) {
      __half2 p = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      r.w[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    return r;
  }
};
template <>
struct Vec<__half, 2> {
  static constexpr int N = 1;
  __device__ __forceinline__ static void widen(const Raw<2>& r, float (&f)[1]) {
    f[0] = __half2float(__ushort_as_half(r.h));
  }
  __device__ __forceinline__ static Raw<2> narrow(const float (&f)[1]) {
    Raw<2> r;
    r.h = __half_as_ushort(__float2half_rn(f[0]));
    return r;
  }
};

template <int VB>
struct Vec<float, VB> {
  static constexpr int N = VB / 4;
  __device__ __forceinline__ static void widen(const Raw<VB>& r, float (&f)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) f[i] = __uint_as_float(r.w[i]);
  }
  __device__ __forceinline__ static Raw<VB> narrow(const float (&f)[N]) {
    Raw<VB> r;
#pragma unroll
    for (int i = 0; i < N; ++i) r.w[i] = __float_as_uint(f[i]);
    return r;
  }
};

// ---------------------------------------------------------------------------
// the arithmetic of the two operations (explicit roundings: no contraction)
// ---------------------------------------------------------------------------

// hidden + update * gate: product rounded, then sum rounded.
__device__ __forceinline__ float residual_gate(float h, float u, float g) {
  return __fadd_rn(h, __fmul_rn(u, g));
}

// n * (1 + scale) + shift with n = x * r, left to right, each op rounded.
__device__ __forceinline__ float modulate(float x, float r, float s, float h) {
  const float n = __fmul_rn(x, r);
  const float one = __fadd_rn(1.0f, s);
  return __fadd_rn(__fmul_rn(n, one), h);
}

// ---------------------------------------------------------------------------
// packed fp32 pairs: float2 with the sm_100 vector intrinsics -- two IEEE
// fp32 operations per instruction, each rounded to nearest-even.  A packed
// multiply whose result feeds a packed add may still be fused into one FMA,
// so where that would change the result the add is a scalar intrinsic.
// ---------------------------------------------------------------------------
using F2 = float2;
__device__ __forceinline__ F2 f2(float lo, float hi) { return make_float2(lo, hi); }
__device__ __forceinline__ float f2_lo(F2 a) { return a.x; }
__device__ __forceinline__ float f2_hi(F2 a) { return a.y; }
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) { return __ffma2_rn(a, b, c); }

// One 32-bit word of storage <-> a pair of fp32 values (bf16x2, half2), or
// one fp32 word <-> one value.
template <class T>
struct Pair;
template <>
struct Pair<__nv_bfloat16> {
  __device__ __forceinline__ static F2 widen(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
  __device__ __forceinline__ static uint32_t narrow(F2 a) {
    __nv_bfloat162 p = __floats2bfloat162_rn(f2_lo(a), f2_hi(a));
    return *reinterpret_cast<uint32_t*>(&p);
  }
};
template <>
struct Pair<__half> {
  __device__ __forceinline__ static F2 widen(uint32_t w) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w));
    return f2(v.x, v.y);
  }
  __device__ __forceinline__ static uint32_t narrow(F2 a) {
    __half2 p = __floats2half2_rn(f2_lo(a), f2_hi(a));
    return *reinterpret_cast<uint32_t*>(&p);
  }
};

// A 16-byte granule as fp32 pairs: 4 pairs of bf16/fp16, 2 pairs of fp32.
template <class T>
struct Granule {
  static constexpr int P = sizeof(T) == 2 ? 4 : 2;
  __device__ __forceinline__ static void widen(const Raw<16>& r, F2 (&f)[P]) {
    if constexpr (sizeof(T) == 2) {
#pragma unroll
      for (int i = 0; i < 4; ++i) f[i] = Pair<T>::widen(r.w[i]);
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i) f[i] = f2(__uint_as_float(r.w[2 * i]), __uint_as_float(r.w[2 * i + 1]));
    }
  }
  __device__ __forceinline__ static Raw<16> narrow(const F2 (&f)[P]) {
    Raw<16> r;
    if constexpr (sizeof(T) == 2) {
#pragma unroll
      for (int i = 0; i < 4; ++i) r.w[i] = Pair<T>::narrow(f[i]);
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        r.w[2 * i] = __float_as_uint(f2_lo(f[i]));
        r.w[2 * i + 1] = __float_as_uint(f2_hi(f[i]));
      }
    }
    return r;
  }
};

// hidden + update * gate on a pair, multiply then add, each rounded to
// nearest, with the scalar non-contractible intrinsics: ptxas fuses a packed
// multiply and a packed add into one FMA (even written with the packed
// intrinsics), and an FMA differs for 16-bit storage too -- a negative
// product below fp32's range added to hidden = +0 gives +0 here and -0 from
// the FMA (found by the test of every bf16 update/gate pair).
template <class T>
__device__ __forceinline__ F2 residual_gate2(F2 h, F2 u, F2 g) {
  return f2(residual_gate(h.x, u.x, g.x), residual_gate(h.y, u.y, g.y));
}

// fl(fl(n * one) + shift) on a pair, n = x * r already formed: the product is
// packed, the final add the non-contractible scalar intrinsic (ptxas
// contracts a packed multiply followed by a packed add into one FMA; the
// bit-exact tests catch it where the add cancels).
__device__ __forceinline__ F2 modulate2(F2 n, F2 one, F2 shift) {
  const F2 t = f2_mul(n, one);
  return f2(__fadd_rn(t.x, shift.x), __fadd_rn(t.y, shift.y));
}

}  // namespace dit
