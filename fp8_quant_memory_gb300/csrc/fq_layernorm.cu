// fq_layernorm.cu -- LayerNorm forward, the fused kernel of "ledger.py" (Ch.13 ledger, layer_norm:
// y = (x - mean) / sqrt(var + eps) * g + b, reading x, g, b once and writing y once).
//
// Cast points (the RMSNorm conventions of the same pages): the row's mean and variance (the mean of
// (x - mean)^2, two passes over the row held on chip, so no E[x^2] - E[x]^2 cancellation) in fp32;
// rstd = 1/sqrt(var + eps), every step correctly rounded; y = dtype(((x - mean) * rstd) * g + b)
// with each fp32 step rounded.
//
// This file: the register-resident kernel (one warp per row, the row's 16-byte vectors in registers,
// for N <= 4096 in the vector layout) and the scalar kernel (any width and alignment). Wide rows on
// >= 4096 rows take the TMA-fed kernel in fq_rows_tma.cu.
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t w32(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// VPT vectors (8 elements each) per lane: vector v = lane + 32 * k.
template <typename T, int VPT>
__global__ void __launch_bounds__(kThreads) ln_vec_kernel(const RowArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int N = a.N, nv = N >> 3;
  const float fN = static_cast<float>(N);
  const T* gp = static_cast<const T*>(a.wq);
  const T* bp = static_cast<const T*>(a.bias);
  const int32_t rows = static_cast<int32_t>(a.rows);
  for (int32_t r = blockIdx.x * kWarps + warp; r < rows; r += gridDim.x * kWarps) {  // warp-uniform
    const T* xrow = static_cast<const T*>(a.x) + static_cast<int64_t>(r) * N;
    uint4 xv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + 32 * k;
      xv[k] = v < nv ? ld_stream16(xrow + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
    }
    // pass 1: mean
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      s0 = add2(s0, add2(Elem<T>::unpack(xv[k].x), Elem<T>::unpack(xv[k].y)));
      s1 = add2(s1, add2(Elem<T>::unpack(xv[k].z), Elem<T>::unpack(xv[k].w)));
    }
    const float2 st = add2(s0, s1);
    const float mean = div_n(group_sum<32>(st.x + st.y), fN);
    const float2 mean2 = splat2(mean);
    // pass 2: variance of the deviations (vectors past the row end hold zeros: not counted)
    float2 q0 = make_float2(0.f, 0.f), q1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (lane + 32 * k >= nv) continue;
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const float2 c0 = sub2(Elem<T>::unpack(w32(xv[k], e)), mean2);
        const float2 c1 = sub2(Elem<T>::unpack(w32(xv[k], e + 1)), mean2);
        q0 = fma2(c0, c0, q0);
        q1 = fma2(c1, c1, q1);
      }
    }
    const float2 qt = add2(q0, q1);
    const float var = div_n(group_sum<32>(qt.x + qt.y), fN);
    const float2 rstd2 = splat2(__frcp_rn(__fsqrt_rn(__fadd_rn(var, a.eps))));
    // pass 3: y
    T* yrow = static_cast<T*>(a.y) + static_cast<int64_t>(r) * N;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = lane + 32 * k;
      if (v >= nv) continue;
      const uint4 gv = ld_cached16(gp + 8 * v);
      const uint4 bv = bp != nullptr ? ld_cached16(bp + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
      uint4 out;
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 c = sub2(Elem<T>::unpack(w32(xv[k], e)), mean2);
        const float2 n = mul2(mul2(c, rstd2), Elem<T>::unpack(w32(gv, e)));
        pk[e] = Elem<T>::pack(add2_rn(n, Elem<T>::unpack(w32(bv, e))));
      }
      out = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      st_stream16(yrow + 8 * v, out);
    }
  }
}

__device__ __forceinline__ float ld1(int dt, const void* p, int64_t i) {
  return dt == DT_BF16 ? Elem<__nv_bfloat16>::load1(p, i) : Elem<__half>::load1(p, i);
}

__global__ void __launch_bounds__(kThreads) ln_scalar_kernel(const RowArgs a, int dt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int N = a.N;
  const float fN = static_cast<float>(N);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + warp; r < a.rows;
       r += static_cast<int64_t>(gridDim.x) * kWarps) {
    float s = 0.f;
    for (int j = lane; j < N; j += 32) s = __fadd_rn(s, ld1(dt, a.x, r * N + j));
    const float mean = div_n(group_sum<32>(s), fN);
    float q = 0.f;
    for (int j = lane; j < N; j += 32) {
      const float c = __fsub_rn(ld1(dt, a.x, r * N + j), mean);
      q = __fmaf_rn(c, c, q);
    }
    const float var = div_n(group_sum<32>(q), fN);
    const float rstd = __frcp_rn(__fsqrt_rn(__fadd_rn(var, a.eps)));
    for (int j = lane; j < N; j += 32) {
      const float c = __fsub_rn(ld1(dt, a.x, r * N + j), mean);
      const float n = __fmul_rn(__fmul_rn(c, rstd), ld1(dt, a.wq, j));
      const float y = __fadd_rn(n, a.bias != nullptr ? ld1(dt, a.bias, j) : 0.f);
      if (dt == DT_BF16) Elem<__nv_bfloat16>::store1(a.y, r * N + j, y);
      else Elem<__half>::store1(a.y, r * N + j, y);
    }
  }
}

template <typename T, int VPT>
void launch_vec(const RowArgs& a, cudaStream_t s) {
  auto kern = ln_vec_kernel<T, VPT>;
  static int per_sm = -1;
  if (per_sm < 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, 0) != cudaSuccess || b < 1) b = 1;
    per_sm = b;
  }
  const int64_t need = (a.rows + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
  kern<<<static_cast<unsigned>(need < cap ? need : cap), kThreads, 0, s>>>(a);
}

template <typename T>
bool dispatch_vec(const RowArgs& a, cudaStream_t s) {
  const int nv = a.N / 8;
  if (nv <= 32) launch_vec<T, 1>(a, s);
  else if (nv <= 64) launch_vec<T, 2>(a, s);
  else if (nv <= 128) launch_vec<T, 4>(a, s);
  else if (nv <= 256) launch_vec<T, 8>(a, s);
  else if (nv <= 512) launch_vec<T, 16>(a, s);
  else return false;
  return true;
}

}  // namespace

void launch_layernorm(const RowArgs& a, int dtype, bool vec, cudaStream_t s) {
  if (vec && launch_layernorm_tma(a, dtype, s)) return;
  if (vec && (dtype == DT_BF16 ? dispatch_vec<__nv_bfloat16>(a, s) : dispatch_vec<__half>(a, s))) return;
  const int64_t need = (a.rows + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  ln_scalar_kernel<<<static_cast<unsigned>(need < cap ? need : cap), kThreads, 0, s>>>(a, dtype);
}

}  // namespace fq
