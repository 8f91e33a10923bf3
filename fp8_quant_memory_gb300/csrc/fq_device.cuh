// fq_device.cuh -- device-side building blocks of the sm_103a kernels: storage-format traits,
// cache-hinted 16/8-byte memory access, packed f32x2 arithmetic, e4m3fn packing, group reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fq {

// ------------------------------------------------------------------------------------------------
// Storage element traits: two packed 16-bit elements (lower address in the low half) <-> float2.
// Conversions to float are exact; conversions from float round to nearest even.
// ------------------------------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  }
  static __device__ __forceinline__ uint32_t pack(float2 v) {
    __nv_bfloat162 h = __float22bfloat162_rn(v);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float load1(const void* p, int64_t i) {
    const uint16_t b = static_cast<const uint16_t*>(p)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    static_cast<__nv_bfloat16*>(p)[i] = h;
  }
};

template <>
struct Elem<__half> {
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return __half22float2(*reinterpret_cast<__half2*>(&u));
  }
  static __device__ __forceinline__ uint32_t pack(float2 v) {
    __half2 h = __float22half2_rn(v);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float load1(const void* p, int64_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float v) {
    static_cast<__half*>(p)[i] = __float2half_rn(v);
  }
};

template <>
struct Elem<float> {
  static __device__ __forceinline__ float load1(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
  }
};

// The same conversions as Elem<T>::unpack, written in PTX. A kernel that needs a packed vector
// unpacked twice (before and after a reduction) uses this for the second time: the compiler cannot
// merge it with the first, so the first set of floats dies early instead of occupying registers.
template <typename T>
__device__ __forceinline__ float2 unpack_again(uint32_t u);

template <>
__device__ __forceinline__ float2 unpack_again<__nv_bfloat16>(uint32_t u) {
  float lo, hi;
  asm("shl.b32 %0, %2, 16;\n\tand.b32 %1, %2, 0xffff0000;" : "=f"(lo), "=f"(hi) : "r"(u));
  return make_float2(lo, hi);
}

template <>
__device__ __forceinline__ float2 unpack_again<__half>(uint32_t u) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(u));
  return make_float2(lo, hi);
}

// Products of 16-bit storage operands rounded once to fp32 (fma.rn.f32.{bf16,f16}: sm_100 and
// later). Two packed elements (low half first) per call.
template <typename T>
struct Mixed;

template <>
struct Mixed<__nv_bfloat16> {
  // (x0*w0, x1*w1), exact: the product of two 8-bit significands fits fp32; -0 + p keeps p's sign.
  static __device__ __forceinline__ float2 mul(uint32_t x, uint32_t w) {
    float2 r;
    asm("{\n\t.reg .b16 x0, x1, w0, w1;\n\tmov.b32 {x0, x1}, %2;\n\tmov.b32 {w0, w1}, %3;\n\t"
        "fma.rn.f32.bf16 %0, x0, w0, %4;\n\tfma.rn.f32.bf16 %1, x1, w1, %4;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(x), "r"(w), "f"(-0.0f));
    return r;
  }
  // (a.x + x0^2, a.y + x1^2)
  static __device__ __forceinline__ float2 sq_add(uint32_t x, float2 a) {
    float2 r;
    asm("{\n\t.reg .b16 x0, x1;\n\tmov.b32 {x0, x1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, x0, x0, %3;\n\tfma.rn.f32.bf16 %1, x1, x1, %4;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(x), "f"(a.x), "f"(a.y));
    return r;
  }
  // (a.x + x0, a.y + x1) rounded once each, as an fp32 add of the unpacked values: x * 1 is exact,
  // and an exact zero sum takes the sign the addition gives it.
  static __device__ __forceinline__ float2 add(uint32_t x, float2 a) {
    float2 r;
    asm("{\n\t.reg .b16 x0, x1, one;\n\tmov.b32 {x0, x1}, %2;\n\tmov.b16 one, 0x3F80;\n\t"
        "fma.rn.f32.bf16 %0, x0, one, %3;\n\tfma.rn.f32.bf16 %1, x1, one, %4;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(x), "f"(a.x), "f"(a.y));
    return r;
  }
};

template <>
struct Mixed<__half> {
  static __device__ __forceinline__ float2 mul(uint32_t x, uint32_t w) {
    float2 r;
    asm("{\n\t.reg .b16 x0, x1, w0, w1;\n\tmov.b32 {x0, x1}, %2;\n\tmov.b32 {w0, w1}, %3;\n\t"
        "fma.rn.f32.f16 %0, x0, w0, %4;\n\tfma.rn.f32.f16 %1, x1, w1, %4;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(x), "r"(w), "f"(-0.0f));
    return r;
  }
  static __device__ __forceinline__ float2 sq_add(uint32_t x, float2 a) {
    float2 r;
    asm("{\n\t.reg .b16 x0, x1;\n\tmov.b32 {x0, x1}, %2;\n\t"
        "fma.rn.f32.f16 %0, x0, x0, %3;\n\tfma.rn.f32.f16 %1, x1, x1, %4;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(x), "f"(a.x), "f"(a.y));
    return r;
  }
  static __device__ __forceinline__ float2 add(uint32_t x, float2 a) {
    float2 r;
    asm("{\n\t.reg .b16 x0, x1, one;\n\tmov.b32 {x0, x1}, %2;\n\tmov.b16 one, 0x3C00;\n\t"
        "fma.rn.f32.f16 %0, x0, one, %3;\n\tfma.rn.f32.f16 %1, x1, one, %4;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(x), "f"(a.x), "f"(a.y));
    return r;
  }
};

// Round a float2 to the storage format and back (the `.to(dtype)` cast of the definition).
template <typename T>
__device__ __forceinline__ float2 round_trip(float2 v) {
  return Elem<T>::unpack(Elem<T>::pack(v));
}

// ------------------------------------------------------------------------------------------------
// Memory access. Streamed data (x, grad_y) bypasses L1 allocation; outputs use evict-first stores.
// Small reused data (weights, rotary tables) goes through the default cached path.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_cached16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ float4 ld_cached16f(const void* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ------------------------------------------------------------------------------------------------
// Packed fp32 pairs (one FFMA2/FMUL2/FADD2 instruction per pair on sm_100-class SMs).
// Each component is rounded exactly like the scalar IEEE operation.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }
// a - b per component (sub.rn.f32x2: one instruction, no separate negation).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }
// a + b per component as its own rounded instruction (inline PTX: never fused with a preceding
// product into an FMA, which would round once where the definition rounds twice).
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  float2 d;
  asm volatile("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Quotient y / s rounded to nearest, given r = RN(1/s) (correctly rounded reciprocal):
// q0 = RN(y*r) is within one ulp of y/s, the residual y - q0*s is exact in one FMA, and
// RN(q0 + residual*r) is the correctly rounded quotient (Markstein's correction, IBM J. Res.
// Dev. 34(1), 1990; Muller et al., Handbook of Floating-Point Arithmetic, ch. 4).
// The correction step turns y = -0 into +0 (+0 + -0 rounds to +0), while the definition's y / s
// keeps the sign of zero (and e4m3fn codes it as 0x80); every other quotient already has the sign
// of y, so copying that sign back is exact.
__device__ __forceinline__ float2 div2_by(float2 y, float s, float r) {
  const float2 q0 = mul2(y, splat2(r));
  const float2 e = fma2(q0, splat2(-s), y);  // y - q0*s, exact: (-q0)*s == q0*(-s)
  const float2 q = fma2(e, splat2(r), q0);
  return make_float2(copysignf(q.x, y.x), copysignf(q.y, y.y));
}

// ------------------------------------------------------------------------------------------------
// e4m3fn: cvt.rn.satfinite rounds to nearest even and saturates at +-448 (the format's largest
// finite value), which is the clamp-then-round of the definition when fp8_max = 448.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2(float2 v) {  // v.x -> low byte, v.y -> high byte
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(v.y), "f"(v.x));
  return d;
}

// 4 quotients -> 4 codes in one word (a.x in the lowest byte). The two 16-bit halves are joined in
// the same inline block as the conversions: measured one instruction per word less than shifting
// and or-ing two zero-extended halves.
__device__ __forceinline__ uint32_t e4m3x4(float2 a, float2 b) {
  uint32_t d;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(d)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// 8 quotients -> 8 codes (element 0 at the lowest address).
__device__ __forceinline__ uint2 pack_e4m3x8(float2 a, float2 b, float2 c, float2 d) {
  return make_uint2(e4m3x4(a, b), e4m3x4(c, d));
}

__device__ __forceinline__ float clamp_abs(float v, float m) { return fminf(fmaxf(v, -m), m); }

// ------------------------------------------------------------------------------------------------
// Reductions over a group of G consecutive lanes (G a power of two <= 32). Every lane of the warp
// must call these (full-mask shuffles); each lane receives its own group's result.
// ------------------------------------------------------------------------------------------------
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float absmax4(float m, float2 a, float2 b) {
  // three-input max.f32 (sm_100+): two instructions for four values
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(fabsf(a.x)), "f"(fabsf(a.y)));
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(r), "f"(fabsf(b.x)), "f"(fabsf(b.y)));
  return r;
}

// x / n correctly rounded, for a row length n >= 1. When n is a power of two, 1/n is exact and x * (1/n)
// is the same real number as x / n, so one rounded product gives the quotient bit for bit (subnormal
// results included); other lengths take the IEEE division.
__device__ __forceinline__ float div_n(float x, float n) {
  const uint32_t b = __float_as_uint(n);
  return (b & 0x7fffffu) == 0u ? __fmul_rn(x, __uint_as_float(0x7f000000u - b)) : __fdiv_rn(x, n);
}

// rstd from the row's sum of squares: 1/sqrt(ss/N + eps), every step correctly rounded in fp32 (the
// correctly rounded reciprocal is the IEEE quotient 1/s). Used where an FP8 code or a saved rstd
// depends on it.
__device__ __forceinline__ float rstd_from_ss(float ss, float n, float eps) {
  return __frcp_rn(__fsqrt_rn(__fadd_rn(div_n(ss, n), eps)));
}

// The same with the hardware reciprocal square root and the approximate quotient (each within 2 ulp
// for the normal range), the pages' rsqrt read as the hardware instruction: a few fp32 ulps from
// rstd_from_ss, far inside the storage-dtype tolerance of the outputs that use it (y of RMSNorm +
// RoPE without quantisation, dx and dw of the backward). About thirty instructions shorter, which
// counts on narrow rows (a 192-element row is 24 elements per lane).
__device__ __forceinline__ float rstd_approx(float ss, float n, float eps) {
  return rsqrtf(__fadd_rn(__fdividef(ss, n), eps));
}

}  // namespace fq
