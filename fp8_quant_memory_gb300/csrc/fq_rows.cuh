// fq_rows.cuh -- per-row arithmetic shared by the row kernels (global-memory and TMA-fed): the
// lane-group layout of a row's 16-byte vectors, and everything from the loaded x vectors to y, the
// scale and the codes.
//
// Definitions: "rmsnorm_rope_quant.py" (Ch.13 fusion), torch_reference_fused / _torch_rope_neox;
// "rmsnorm_tl.py" (Ch.17), _rmsnorm_fwd; "case_norm_rope_quant.py" (Ch.28), the prologue.
#pragma once

#include "fq_device.cuh"
#include "fq_internal.h"

namespace fq {
namespace rows {

__device__ __forceinline__ uint32_t word(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

__device__ __forceinline__ void set_word(uint4& v, int k, uint32_t u) {
  if (k == 0) v.x = u;
  else if (k == 1) v.y = u;
  else if (k == 2) v.z = u;
  else v.w = u;
}

// 8 consecutive table entries starting at element `off` -> 4 float2 (entries 2k, 2k+1 in [k]).
// SMEM: `base` points into shared memory (a staged table block) instead of global memory.
template <typename TT, bool SMEM>
__device__ __forceinline__ void load_table8(const void* base, int64_t off, float2 (&v)[4]) {
  if constexpr (SMEM) {
    const TT* p = static_cast<const TT*>(base) + off;
    if constexpr (sizeof(TT) == 4) {
      const float4 a = *reinterpret_cast<const float4*>(p);
      const float4 b = *reinterpret_cast<const float4*>(p + 4);
      v[0] = make_float2(a.x, a.y);
      v[1] = make_float2(a.z, a.w);
      v[2] = make_float2(b.x, b.y);
      v[3] = make_float2(b.z, b.w);
    } else {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      v[0] = Elem<TT>::unpack(u.x);
      v[1] = Elem<TT>::unpack(u.y);
      v[2] = Elem<TT>::unpack(u.z);
      v[3] = Elem<TT>::unpack(u.w);
    }
    return;
  }
  if constexpr (sizeof(TT) == 4) {
    const float* p = static_cast<const float*>(base) + off;
    const float4 a = ld_cached16f(p);
    const float4 b = ld_cached16f(p + 4);
    v[0] = make_float2(a.x, a.y);
    v[1] = make_float2(a.z, a.w);
    v[2] = make_float2(b.x, b.y);
    v[3] = make_float2(b.z, b.w);
  } else {
    const uint4 u = ld_cached16(static_cast<const TT*>(base) + off);
    v[0] = Elem<TT>::unpack(u.x);
    v[1] = Elem<TT>::unpack(u.y);
    v[2] = Elem<TT>::unpack(u.z);
    v[3] = Elem<TT>::unpack(u.w);
  }
}

// Column of the first element of vector slot s of lane `lane`, and whether that slot exists in a row
// (slots: HS head vectors, TS tail-lo vectors, TS tail-hi vectors). s is a compile-time constant in
// every caller, so both fold into an immediate offset and one compare.
template <int LPR, int HS, int TS>
__device__ __forceinline__ int slot_col(int s, int lane, int hv, int th) {
  if (s < HS) return 8 * (lane + s * LPR);
  if (s < HS + TS) return 8 * (hv + lane + (s - HS) * LPR);
  return 8 * (hv + th + lane + (s - HS - TS) * LPR);
}

template <int LPR, int HS, int TS>
__device__ __forceinline__ bool slot_ok(int s, int lane, int hv, int th) {
  if (s < HS) return lane + s * LPR < hv;
  return lane + ((s - HS) % (TS > 0 ? TS : 1)) * LPR < th;
}

// Everything after the loads for one row held by a lane group: rstd, normalise, rotate, write y
// (fwd / rope modes write each vector as soon as it is computed), amax, scale, codes.
// Group-wise scales (MODE_ROPE_QUANT with a.group > 0, "rms_norm_rope_quant_fused" step 3): `gmax`
// is this row's array of N / a.group words in shared memory; each lane folds its slots' |y| maxima
// into their groups with atomicMax on the float bits (non-negative floats order like their bits),
// and quantises each slot with its own group's scale. A 16-byte vector never straddles a group
// (a.group % 8 == 0).
// Table entries of this row: cos_base/sin_base + trow + pair index (global memory, or a staged block
// in shared memory when SMEM_TAB). WPRE: the caller holds this lane's weight vectors in `wpre` (one
// per slot, loaded once for every row it processes; single-weight modes only), else they are read
// from global memory per row.
template <typename T, typename TT, int MODE, int LPR, int HS, int TS, bool SMEM_TAB, bool WPRE = false>
__device__ __forceinline__ void row_body(const RowArgs& a, int32_t r, bool rv, int32_t h,
                                         const uint4 (&xv)[HS + 2 * TS], int lane, int hv, int th, float fN,
                                         const void* cos_base, const void* sin_base, int64_t trow,
                                         const uint4* wpre = nullptr, uint32_t* gmax = nullptr) {
  static_assert(!(WPRE && MODE == MODE_QK), "the prologue selects wq or wk per row");
  constexpr bool kQuant = (MODE == MODE_ROPE_QUANT) || (MODE == MODE_QK);
  constexpr bool kRound = (MODE == MODE_ROPE) || (MODE == MODE_ROPE_QUANT);
  constexpr int kV = HS + 2 * TS;  // vector slots per lane: head..., tail-lo..., tail-hi...
  const int N = a.N;

  // a2: sum of squares -> rstd, the squares taken straight from the 16-bit storage operands (x*x of a
  // 16-bit value is exact in fp32 and each FMA rounds once, as an FMA on the unpacked values does:
  // the same sums without unpacking x). RMSNorm + RoPE without quantisation (MODE_ROPE) also
  // normalises as (x * w) * rstd with x * w exact: the same values as (x * rstd) * w up to one fp32
  // rounding, the size of the approximate rstd this mode already uses, and no unpacking of x or w.
  constexpr bool kMixed = MODE == MODE_ROPE;
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int s = 0; s < kV; ++s) {
    acc0 = Mixed<T>::sq_add(xv[s].x, acc0);
    acc1 = Mixed<T>::sq_add(xv[s].y, acc1);
    acc0 = Mixed<T>::sq_add(xv[s].z, acc0);
    acc1 = Mixed<T>::sq_add(xv[s].w, acc1);
  }
  const float2 acc = add2(acc0, acc1);
  const float ss = group_sum<LPR>(acc.x + acc.y);
  const float rstd = MODE == MODE_ROPE ? rstd_approx(ss, fN, a.eps) : rstd_from_ss(ss, fN, a.eps);
  if (MODE == MODE_FWD && a.rstd != nullptr && rv && lane == 0) a.rstd[r] = rstd;
  const float2 rstd2 = splat2(rstd);
  const T* wrow = static_cast<const T*>((MODE == MODE_QK && h >= a.Hq) ? a.wk : a.wq);
  T* yrow = (MODE != MODE_QK && a.y != nullptr && rv) ? static_cast<T*>(a.y) + static_cast<int64_t>(r) * N
                                                      : nullptr;

  uint4 yp[kV];      // rounded y kept for the quantiser (MODE_ROPE_QUANT)
  float2 yf[kV][4];  // fp32 y kept for the quantiser (MODE_QK)
  float ams[kV];     // per-slot |y| maxima (group-wise scales)
  float amax = 0.f;

  // a3: head columns, normalised (rounded to the storage dtype unless MODE_QK)
#pragma unroll
  for (int s = 0; s < HS; ++s) {
    ams[s] = 0.f;
    if (!slot_ok<LPR, HS, TS>(s, lane, hv, th)) {
      yp[s] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int k = 0; k < 4; ++k) yf[s][k] = make_float2(0.f, 0.f);
      continue;
    }
    const uint4 wv = WPRE ? wpre[s] : ld_cached16(wrow + slot_col<LPR, HS, TS>(s, lane, hv, th));
    uint4 packed;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 n = kMixed ? mul2(Mixed<T>::mul(word(xv[s], k), word(wv, k)), rstd2)
                              : mul2(mul2(Elem<T>::unpack(word(xv[s], k)), rstd2), Elem<T>::unpack(word(wv, k)));
      if constexpr (MODE == MODE_QK) {
        yf[s][k] = n;
      } else {
        const uint32_t pk = Elem<T>::pack(n);
        set_word(packed, k, pk);
        if constexpr (kQuant) {
          const float2 rn = Elem<T>::unpack(pk);
          ams[s] = fmaxf(ams[s], fmaxf(fabsf(rn.x), fabsf(rn.y)));
        }
      }
    }
    if constexpr (MODE == MODE_QK) {
      amax = absmax4(absmax4(amax, yf[s][0], yf[s][1]), yf[s][2], yf[s][3]);
    } else {
      if (yrow != nullptr) st_stream16(yrow + slot_col<LPR, HS, TS>(s, lane, hv, th), packed);
      if constexpr (kQuant) {
        yp[s] = packed;
        amax = fmaxf(amax, ams[s]);
      }
    }
  }

  // a4: rotary pairs
  if constexpr (TS > 0) {
#pragma unroll
    for (int s = 0; s < TS; ++s) {
      const int slo = HS + s, shi = HS + TS + s;
      ams[slo] = ams[shi] = 0.f;
      if (!slot_ok<LPR, HS, TS>(slo, lane, hv, th)) {
        yp[slo] = yp[shi] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k) yf[slo][k] = yf[shi][k] = make_float2(0.f, 0.f);
        continue;
      }
      const int p8 = 8 * (lane + s * LPR);  // pair index of the vector's first element
      const uint4 wlo = WPRE ? wpre[slo] : ld_cached16(wrow + slot_col<LPR, HS, TS>(slo, lane, hv, th));
      const uint4 whi = WPRE ? wpre[shi] : ld_cached16(wrow + slot_col<LPR, HS, TS>(shi, lane, hv, th));
      float2 c[4], sn[4];
      load_table8<TT, SMEM_TAB>(cos_base, trow + p8, c);
      load_table8<TT, SMEM_TAB>(sin_base, trow + p8, sn);
      uint4 plo4, phi4;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 lo = kMixed ? mul2(Mixed<T>::mul(word(xv[slo], k), word(wlo, k)), rstd2)
                           : mul2(mul2(Elem<T>::unpack(word(xv[slo], k)), rstd2), Elem<T>::unpack(word(wlo, k)));
        float2 hi = kMixed ? mul2(Mixed<T>::mul(word(xv[shi], k), word(whi, k)), rstd2)
                           : mul2(mul2(Elem<T>::unpack(word(xv[shi], k)), rstd2), Elem<T>::unpack(word(whi, k)));
        if constexpr (kRound) {
          lo = round_trip<T>(lo);
          hi = round_trip<T>(hi);
        }
        const float2 ylo = sub2(mul2(lo, c[k]), mul2(hi, sn[k]));
        const float2 yhi = add2(mul2(hi, c[k]), mul2(lo, sn[k]));
        if constexpr (MODE == MODE_QK) {
          yf[slo][k] = ylo;
          yf[shi][k] = yhi;
        } else {
          const uint32_t plo = Elem<T>::pack(ylo), phi = Elem<T>::pack(yhi);
          set_word(plo4, k, plo);
          set_word(phi4, k, phi);
          if constexpr (kQuant) {
            const float2 rl = Elem<T>::unpack(plo), rh = Elem<T>::unpack(phi);
            ams[slo] = fmaxf(ams[slo], fmaxf(fabsf(rl.x), fabsf(rl.y)));
            ams[shi] = fmaxf(ams[shi], fmaxf(fabsf(rh.x), fabsf(rh.y)));
          }
        }
      }
      if constexpr (MODE == MODE_QK) {
        amax = absmax4(absmax4(amax, yf[slo][0], yf[slo][1]), yf[slo][2], yf[slo][3]);
        amax = absmax4(absmax4(amax, yf[shi][0], yf[shi][1]), yf[shi][2], yf[shi][3]);
      } else {
        if (yrow != nullptr) {
          st_stream16(yrow + slot_col<LPR, HS, TS>(slo, lane, hv, th), plo4);
          st_stream16(yrow + slot_col<LPR, HS, TS>(shi, lane, hv, th), phi4);
        }
        if constexpr (kQuant) {
          yp[slo] = plo4;
          yp[shi] = phi4;
          amax = fmaxf(amax, fmaxf(ams[slo], ams[shi]));
        }
      }
    }
  }

  // a6-a8 with group-wise scales
  if constexpr (MODE == MODE_ROPE_QUANT) {
    if (gmax != nullptr) {
      const int gs = a.group, G = N / gs;
      __syncwarp();  // the previous row's readers of this array are done
      for (int g = lane; g < G; g += LPR) gmax[g] = 0u;
      __syncwarp();
#pragma unroll
      for (int s = 0; s < kV; ++s)
        if (slot_ok<LPR, HS, TS>(s, lane, hv, th))
          atomicMax(&gmax[slot_col<LPR, HS, TS>(s, lane, hv, th) / gs], __float_as_uint(ams[s]));
      __syncwarp();
      if (rv) {
        const bool clamp = a.fp8_max != 448.0f;
        uint8_t* qrow = a.q + static_cast<int64_t>(r) * N;
#pragma unroll
        for (int s = 0; s < kV; ++s) {
          if (!slot_ok<LPR, HS, TS>(s, lane, hv, th)) continue;
          const int col = slot_col<LPR, HS, TS>(s, lane, hv, th);
          const float sc = __fdiv_rn(fmaxf(__uint_as_float(gmax[col / gs]), 1e-4f), a.fp8_max);
          const float rc = __frcp_rn(sc);
          float2 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[k] = div2_by(Elem<T>::unpack(word(yp[s], k)), sc, rc);
            if (clamp) v[k] = make_float2(clamp_abs(v[k].x, a.fp8_max), clamp_abs(v[k].y, a.fp8_max));
          }
          st_stream8(qrow + col, pack_e4m3x8(v[0], v[1], v[2], v[3]));
        }
        for (int g = lane; g < G; g += LPR)
          a.scale[static_cast<int64_t>(r) * G + g] = __fdiv_rn(fmaxf(__uint_as_float(gmax[g]), 1e-4f), a.fp8_max);
      }
      return;
    }
  }

  // a6-a8: scale and codes
  if constexpr (kQuant) {
    amax = fmaxf(group_max<LPR>(amax), 1e-4f);
    const float sc = __fdiv_rn(amax, a.fp8_max);
    const float rc = __frcp_rn(sc);
    const bool clamp = a.fp8_max != 448.0f;
    if (rv) {
      uint8_t* qrow = a.q + static_cast<int64_t>(r) * N;
#pragma unroll
      for (int s = 0; s < kV; ++s) {
        if (!slot_ok<LPR, HS, TS>(s, lane, hv, th)) continue;
        float2 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 yy = (MODE == MODE_QK) ? yf[s][k] : Elem<T>::unpack(word(yp[s], k));
          v[k] = div2_by(yy, sc, rc);
          if (clamp) v[k] = make_float2(clamp_abs(v[k].x, a.fp8_max), clamp_abs(v[k].y, a.fp8_max));
        }
        st_stream8(qrow + slot_col<LPR, HS, TS>(s, lane, hv, th), pack_e4m3x8(v[0], v[1], v[2], v[3]));
      }
      if (lane == 0) a.scale[r] = sc;
    }
  }
}

}  // namespace rows
}  // namespace fq
