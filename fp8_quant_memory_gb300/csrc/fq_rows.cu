// fq_rows.cu -- vectorised row kernel for RMSNorm, RMSNorm+RoPE, RMSNorm+RoPE+FP8 and the
// QK-Norm+RoPE+FP8 prologue.
//
// Definitions: "rmsnorm_rope_quant.py" (Ch.13 fusion), torch_reference_fused / _torch_rope_neox;
// "rmsnorm_tl.py" (Ch.17), _rmsnorm_fwd; "case_norm_rope_quant.py" (Ch.28), the prologue.
//
// Layout of the work: a group of LPR consecutive lanes owns one row. Lane l of the group holds
//   - head vectors (8 elements, 16 bytes each) l, l+LPR, ... of the N-R unrotated columns, and
//   - rotary pairs of vectors: the tail's first-half vector p = l, l+LPR, ... together with its
//     partner p + R/16 in the second half,
// so each NeoX pair (j, j+R/2) sits in one thread's registers: no shuffle and no shared-memory
// round trip for the rotation (the TileLang kernels of the fusion page stage the row through shared
// memory for exactly this pairing). Loads of a group still cover contiguous 16-byte runs.
// x is read once with L1::no_allocate; weight vectors and table rows go through L1, which serves
// the other rows of the same token (the prologue's table is per token, per Ch.28 design C).
// Reductions (sum of squares, amax) are group shuffles.
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fq {
namespace {

constexpr int kThreads = 256;

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
template <typename TT>
__device__ __forceinline__ void load_table8(const void* base, int64_t off, float2 (&v)[4]) {
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

template <typename T, typename TT, int MODE, int LPR, int HS, int TS>
__global__ void __launch_bounds__(kThreads) rows_vec_kernel(const RowArgs a) {
  constexpr bool kQuant = (MODE == MODE_ROPE_QUANT) || (MODE == MODE_QK);
  constexpr bool kRound = (MODE == MODE_ROPE) || (MODE == MODE_ROPE_QUANT);
  constexpr int kRowsPerCta = kThreads / LPR;
  constexpr int kV = HS + 2 * TS;  // vector slots per lane: head..., tail-lo..., tail-hi...

  const int lane = threadIdx.x & (LPR - 1);
  const int grp = threadIdx.x / LPR;
  const int N = a.N;
  const int hv = (N - a.R) >> 3;  // head vectors
  const int th = a.R >> 4;        // rotary pairs of vectors
  const int half = a.R >> 1;
  const float fN = static_cast<float>(N);

  int col[kV];
  bool ok[kV];
#pragma unroll
  for (int s = 0; s < HS; ++s) {
    const int v = lane + s * LPR;
    col[s] = 8 * v;
    ok[s] = v < hv;
  }
#pragma unroll
  for (int s = 0; s < TS; ++s) {
    const int p = lane + s * LPR;
    col[HS + s] = 8 * (hv + p);
    col[HS + TS + s] = 8 * (hv + th + p);
    ok[HS + s] = ok[HS + TS + s] = p < th;
  }

  const int32_t rows = static_cast<int32_t>(a.rows);
  for (int32_t base = blockIdx.x * kRowsPerCta; base < rows; base += gridDim.x * kRowsPerCta) {
    const int32_t r = base + grp;
    const bool rv = r < rows;
    int32_t t = r, h = 0;
    if constexpr (MODE == MODE_QK) {
      t = r / a.H;
      h = r - t * a.H;
    }
    const T* xrow = static_cast<const T*>(a.x) + (static_cast<int64_t>(t) * a.token_stride +
                                                    static_cast<int64_t>(h) * N);
    uint4 xv[kV];
#pragma unroll
    for (int s = 0; s < kV; ++s)
      xv[s] = (rv && ok[s]) ? ld_stream16(xrow + col[s]) : make_uint4(0u, 0u, 0u, 0u);

    // a2: sum of squares -> rstd
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kV; ++s)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = Elem<T>::unpack(word(xv[s], k));
        acc = fma2(f, f, acc);
      }
    const float ss = group_sum<LPR>(acc.x + acc.y);
    const float rstd = rstd_from_ss(ss, fN, a.eps);
    const float2 rstd2 = splat2(rstd);
    const T* wrow = static_cast<const T*>((MODE == MODE_QK && h >= a.Hq) ? a.wk : a.wq);

    uint4 yp[kV];       // rounded y (storage dtype), kRound and MODE_FWD
    float2 yf[kV][4];   // fp32 y, MODE_QK
    float amax = 0.f;

    // a3: head columns, normalised (and rounded unless MODE_QK)
#pragma unroll
    for (int s = 0; s < HS; ++s) {
      if (!ok[s]) {
        yp[s] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k) yf[s][k] = make_float2(0.f, 0.f);
        continue;
      }
      const uint4 wv = ld_cached16(wrow + col[s]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 n = mul2(mul2(Elem<T>::unpack(word(xv[s], k)), rstd2), Elem<T>::unpack(word(wv, k)));
        if constexpr (MODE == MODE_QK) {
          yf[s][k] = n;
        } else {
          const uint32_t pk = Elem<T>::pack(n);
          set_word(yp[s], k, pk);
          if constexpr (kQuant) {
            const float2 rn = Elem<T>::unpack(pk);
            amax = absmax4(amax, rn, make_float2(0.f, 0.f));
          }
        }
      }
      if constexpr (MODE == MODE_QK) amax = absmax4(absmax4(amax, yf[s][0], yf[s][1]), yf[s][2], yf[s][3]);
    }

    // a4: rotary pairs
    if constexpr (TS > 0) {
      const int64_t trow = static_cast<int64_t>(t) * half;
#pragma unroll
      for (int s = 0; s < TS; ++s) {
        const int slo = HS + s, shi = HS + TS + s;
        if (!ok[slo]) {
          yp[slo] = yp[shi] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int k = 0; k < 4; ++k) yf[slo][k] = yf[shi][k] = make_float2(0.f, 0.f);
          continue;
        }
        const int p8 = 8 * (lane + s * LPR);  // pair index of the vector's first element
        const uint4 wlo = ld_cached16(wrow + col[slo]);
        const uint4 whi = ld_cached16(wrow + col[shi]);
        float2 c[4], sn[4];
        load_table8<TT>(a.cos, trow + p8, c);
        load_table8<TT>(a.sin, trow + p8, sn);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float2 lo = mul2(mul2(Elem<T>::unpack(word(xv[slo], k)), rstd2), Elem<T>::unpack(word(wlo, k)));
          float2 hi = mul2(mul2(Elem<T>::unpack(word(xv[shi], k)), rstd2), Elem<T>::unpack(word(whi, k)));
          if constexpr (kRound) {
            lo = round_trip<T>(lo);
            hi = round_trip<T>(hi);
          }
          float2 ylo = sub2(mul2(lo, c[k]), mul2(hi, sn[k]));
          float2 yhi = add2(mul2(hi, c[k]), mul2(lo, sn[k]));
          if constexpr (MODE == MODE_QK) {
            yf[slo][k] = ylo;
            yf[shi][k] = yhi;
          } else {
            const uint32_t plo = Elem<T>::pack(ylo), phi = Elem<T>::pack(yhi);
            set_word(yp[slo], k, plo);
            set_word(yp[shi], k, phi);
            if constexpr (kQuant) amax = absmax4(amax, Elem<T>::unpack(plo), Elem<T>::unpack(phi));
          }
        }
        if constexpr (MODE == MODE_QK) {
          amax = absmax4(absmax4(amax, yf[slo][0], yf[slo][1]), yf[slo][2], yf[slo][3]);
          amax = absmax4(absmax4(amax, yf[shi][0], yf[shi][1]), yf[shi][2], yf[shi][3]);
        }
      }
    }

    // a5: y
    if constexpr (MODE != MODE_QK) {
      if (a.y != nullptr && rv) {
        T* yrow = static_cast<T*>(a.y) + static_cast<int64_t>(r) * N;
#pragma unroll
        for (int s = 0; s < kV; ++s)
          if (ok[s]) st_stream16(yrow + col[s], yp[s]);
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
          if (!ok[s]) continue;
          float2 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 yy = (MODE == MODE_QK) ? yf[s][k] : Elem<T>::unpack(word(yp[s], k));
            v[k] = div2_by(yy, sc, rc);
            if (clamp) v[k] = make_float2(clamp_abs(v[k].x, a.fp8_max), clamp_abs(v[k].y, a.fp8_max));
          }
          st_stream8(qrow + col[s], pack_e4m3x8(v[0], v[1], v[2], v[3]));
        }
        if (lane == 0) a.scale[r] = sc;
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Instantiation table. (LPR, HS, TS) must cover hv = (N-R)/8 <= LPR*HS and th = R/16 <= LPR*TS.
// ------------------------------------------------------------------------------------------------
struct Shape {
  int lpr, hs, ts;
};

template <typename T, typename TT, int MODE, int LPR, int HS, int TS>
bool launch_one(const RowArgs& a, cudaStream_t s) {
  auto kern = rows_vec_kernel<T, TT, MODE, LPR, HS, TS>;
  static int blocks_per_sm = -1;
  if (blocks_per_sm < 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, 0) != cudaSuccess || b < 1) b = 1;
    blocks_per_sm = b;
  }
  constexpr int kRowsPerCta = kThreads / LPR;
  const int64_t need = (a.rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm;
  const int grid = static_cast<int>(need < cap ? need : cap);
  kern<<<grid, kThreads, 0, s>>>(a);
  return true;
}

#define FQ_SHAPES(X)          \
  X(8, 0, 1) X(8, 2, 1) X(16, 2, 1) X(32, 2, 1) X(32, 4, 1) X(32, 8, 1) X(32, 16, 1)
#define FQ_SHAPES_NOROPE(X) \
  X(8, 1, 0) X(8, 2, 0) X(8, 4, 0) X(16, 4, 0) X(32, 4, 0) X(32, 8, 0) X(32, 16, 0)
#define FQ_SHAPES_QK(X) X(8, 0, 1) X(8, 2, 1) X(16, 2, 1) X(32, 2, 1)

template <typename T, typename TT, int MODE>
bool dispatch_shape(const RowArgs& a, cudaStream_t s) {
  const int hv = (a.N - a.R) / 8, th = a.R / 16;
#define FQ_TRY(L, H, S)                                                    \
  if (hv <= (L) * (H) && th <= (L) * (S) && ((S) > 0 || th == 0))          \
    return launch_one<T, TT, MODE, L, H, S>(a, s);
  if constexpr (MODE == MODE_FWD) {
    FQ_SHAPES_NOROPE(FQ_TRY)
  } else if constexpr (MODE == MODE_QK) {
    FQ_SHAPES_QK(FQ_TRY)
  } else {
    if (th == 0) {  // no rotation: the no-rope shapes are cheaper
      FQ_SHAPES_NOROPE(FQ_TRY)
    }
    FQ_SHAPES(FQ_TRY)
  }
#undef FQ_TRY
  return false;
}

template <typename T, int MODE>
bool dispatch_table(const RowArgs& a, int table_dtype, cudaStream_t s) {
  if (MODE == MODE_FWD || a.R == 0) return dispatch_shape<T, T, MODE>(a, s);
  if (table_dtype == DT_FP32) return dispatch_shape<T, float, MODE>(a, s);
  return dispatch_shape<T, T, MODE>(a, s);  // caller checked table_dtype == dtype
}

template <typename T>
bool dispatch_mode(const RowArgs& a, int mode, int table_dtype, cudaStream_t s) {
  switch (mode) {
    case MODE_FWD: return dispatch_table<T, MODE_FWD>(a, table_dtype, s);
    case MODE_ROPE: return dispatch_table<T, MODE_ROPE>(a, table_dtype, s);
    case MODE_ROPE_QUANT: return dispatch_table<T, MODE_ROPE_QUANT>(a, table_dtype, s);
    case MODE_QK: return dispatch_table<T, MODE_QK>(a, table_dtype, s);
  }
  return false;
}

}  // namespace

bool launch_rows_vector(const RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s) {
  if (a.R > 0 && table_dtype != DT_FP32 && table_dtype != dtype) return false;
  if (dtype == DT_BF16) return dispatch_mode<__nv_bfloat16>(a, mode, table_dtype, s);
  if (dtype == DT_FP16) return dispatch_mode<__half>(a, mode, table_dtype, s);
  return false;
}

}  // namespace fq
