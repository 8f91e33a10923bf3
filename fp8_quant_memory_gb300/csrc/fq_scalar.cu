// fq_scalar.cu -- element-wise fallback for the row kernels: any width N, any even rope_dim, any
// pointer alignment and any (storage dtype, table dtype) pair. One warp per row; the row is read
// from global memory once per pass (L1/L2 serve the re-reads). Same arithmetic and cast points as
// the vectorised kernel, with the division done by the IEEE divide.
//
// Definitions: "rmsnorm_rope_quant.py" (Ch.13 fusion), torch_reference_fused; "rmsnorm_tl.py"
// (Ch.17), _rmsnorm_fwd; "case_norm_rope_quant.py" (Ch.28), the prologue.
#include "fq_device.cuh"
#include "fq_internal.h"

namespace fq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float ld_any(int dt, const void* p, int64_t i) {
  if (dt == DT_BF16) return Elem<__nv_bfloat16>::load1(p, i);
  if (dt == DT_FP16) return Elem<__half>::load1(p, i);
  return Elem<float>::load1(p, i);
}

__device__ __forceinline__ float round_any(int dt, float v) {
  if (dt == DT_BF16) return __bfloat162float(__float2bfloat16_rn(v));
  if (dt == DT_FP16) return __half2float(__float2half_rn(v));
  return v;
}

__device__ __forceinline__ void st_any(int dt, void* p, int64_t i, float v) {
  if (dt == DT_BF16) Elem<__nv_bfloat16>::store1(p, i, v);
  else Elem<__half>::store1(p, i, v);
}

__device__ __forceinline__ uint8_t e4m3(float v) {
  return static_cast<uint8_t>(e4m3x2(make_float2(v, 0.f)) & 0xFFu);
}

struct RowCtx {
  const void* x;     // row start
  const void* w;     // weight for this row
  int64_t trow;      // table row offset (elements)
  float rstd;
  int N, R, half;
  int dt, tdt;
  bool round;
};

__device__ __forceinline__ float normed(const RowCtx& c, int j) {
  const float n = __fmul_rn(__fmul_rn(ld_any(c.dt, c.x, j), c.rstd), ld_any(c.dt, c.w, j));
  return c.round ? round_any(c.dt, n) : n;
}

// y_j of the definition: the normalised value, rotated with its NeoX partner in the tail.
__device__ float y_at(const RowCtx& c, const void* cs, const void* sn, int j) {
  const int base = c.N - c.R;
  if (j < base) return normed(c, j);
  int p = j - base;
  const bool first = p < c.half;
  if (!first) p -= c.half;
  const float lo = normed(c, base + p);
  const float hi = normed(c, base + c.half + p);
  const float co = ld_any(c.tdt, cs, c.trow + p);
  const float si = ld_any(c.tdt, sn, c.trow + p);
  const float y = first ? __fsub_rn(__fmul_rn(lo, co), __fmul_rn(hi, si))
                        : __fadd_rn(__fmul_rn(hi, co), __fmul_rn(lo, si));
  return c.round ? round_any(c.dt, y) : y;
}

__global__ void __launch_bounds__(kThreads)
    rows_scalar_kernel(const RowArgs a, int mode, int dt, int tdt) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool quant = (mode == MODE_ROPE_QUANT) || (mode == MODE_QK);
  const int64_t esize = (dt == DT_FP32) ? 4 : 2;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kWarps; base < a.rows;
       base += static_cast<int64_t>(gridDim.x) * kWarps) {
    const int64_t r = base + warp;
    if (r >= a.rows) continue;  // warp-uniform
    int64_t t = r, h = 0;
    if (mode == MODE_QK) {
      t = r / a.H;
      h = r - t * a.H;
    }
    RowCtx c;
    c.x = static_cast<const char*>(a.x) + (t * a.token_stride + h * a.N) * esize;
    c.w = (mode == MODE_QK && h >= a.Hq) ? a.wk : a.wq;
    c.N = a.N;
    c.R = a.R;
    c.half = a.R / 2;
    c.trow = t * c.half;
    c.dt = dt;
    c.tdt = tdt;
    c.round = (mode == MODE_ROPE) || (mode == MODE_ROPE_QUANT);

    float ss = 0.f;
    for (int j = lane; j < a.N; j += 32) {
      const float v = ld_any(dt, c.x, j);
      ss = __fmaf_rn(v, v, ss);
    }
    ss = group_sum<32>(ss);
    c.rstd = rstd_from_ss(ss, static_cast<float>(a.N), a.eps);
    if (mode == MODE_FWD && a.rstd != nullptr && lane == 0) a.rstd[r] = c.rstd;

    if (mode != MODE_QK && a.y != nullptr)
      for (int j = lane; j < a.N; j += 32) {
        const float y = (mode == MODE_FWD) ? __fmul_rn(__fmul_rn(ld_any(dt, c.x, j), c.rstd), ld_any(dt, c.w, j))
                                           : y_at(c, a.cos, a.sin, j);
        st_any(dt, a.y, r * a.N + j, y);
      }
    if (!quant) continue;
    // One scale per group of gs consecutive columns (gs = N: one per row).
    const int gs = (mode == MODE_ROPE_QUANT && a.group > 0) ? a.group : a.N;
    const int G = a.N / gs;
    for (int g = 0; g < G; ++g) {
      float amax = 0.f;
      for (int j = g * gs + lane; j < (g + 1) * gs; j += 32) amax = fmaxf(amax, fabsf(y_at(c, a.cos, a.sin, j)));
      amax = fmaxf(group_max<32>(amax), 1e-4f);
      const float sc = __fdiv_rn(amax, a.fp8_max);
      for (int j = g * gs + lane; j < (g + 1) * gs; j += 32) {
        const float y = y_at(c, a.cos, a.sin, j);
        a.q[r * a.N + j] = e4m3(clamp_abs(__fdiv_rn(y, sc), a.fp8_max));
      }
      if (lane == 0) a.scale[r * G + g] = sc;
    }
  }
}

}  // namespace

void launch_rows_scalar(const RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s) {
  const int64_t need = (a.rows + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int grid = static_cast<int>(need < cap ? need : cap);
  rows_scalar_kernel<<<grid, kThreads, 0, s>>>(a, mode, dtype, table_dtype);
}

}  // namespace fq
