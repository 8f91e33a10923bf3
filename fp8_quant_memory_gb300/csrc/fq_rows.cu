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
#include "fq_rows.cuh"

namespace fq {
namespace {

using namespace rows;

constexpr int kThreads = 256;

// U rows per lane group per iteration: all U rows' loads are issued before any of them is used,
// so a warp keeps U times the bytes in flight (narrow rows need it to cover HBM latency).
template <typename T, typename TT, int MODE, int LPR, int HS, int TS, int U>
__global__ void __launch_bounds__(kThreads) rows_vec_kernel(const RowArgs a) {
  constexpr int kRowsPerCta = kThreads / LPR;
  constexpr int kV = HS + 2 * TS;
  extern __shared__ uint32_t group_max[];  // [kRowsPerCta][N / a.group] with group-wise scales

  const int lane = threadIdx.x & (LPR - 1);
  const int grp = threadIdx.x / LPR;
  const int N = a.N;
  const int hv = (N - a.R) >> 3;  // head vectors
  const int th = a.R >> 4;        // rotary pairs of vectors
  const int half = a.R >> 1;
  const float fN = static_cast<float>(N);

  const int32_t rows = static_cast<int32_t>(a.rows);
  for (int32_t base = blockIdx.x * (kRowsPerCta * U); base < rows; base += gridDim.x * (kRowsPerCta * U)) {
    int32_t r[U], t[U], h[U];
    bool rv[U];
    uint4 xv[U][kV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      r[u] = base + u * kRowsPerCta + grp;
      rv[u] = r[u] < rows;
      t[u] = r[u];
      h[u] = 0;
      if constexpr (MODE == MODE_QK) {
        t[u] = r[u] / a.H;
        h[u] = r[u] - t[u] * a.H;
      }
      const T* xrow = static_cast<const T*>(a.x) + (static_cast<int64_t>(t[u]) * a.token_stride +
                                                      static_cast<int64_t>(h[u]) * N);
#pragma unroll
      for (int s = 0; s < kV; ++s)
        xv[u][s] = (rv[u] && slot_ok<LPR, HS, TS>(s, lane, hv, th))
                       ? ld_stream16(xrow + slot_col<LPR, HS, TS>(s, lane, hv, th))
                       : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t* gmax = (MODE == MODE_ROPE_QUANT && a.group > 0) ? group_max + grp * (N / a.group) : nullptr;
#pragma unroll
    for (int u = 0; u < U; ++u)
      row_body<T, TT, MODE, LPR, HS, TS, false>(a, r[u], rv[u], h[u], xv[u], lane, hv, th, fN, a.cos, a.sin,
                                                static_cast<int64_t>(t[u]) * half, nullptr, gmax);
  }
}

// The Ch.28 page's designs A / B / C ("case_norm_rope_quant.py", default_designs): one CTA per block
// of `rpb` consecutive (token, head) rows -- 1 (A), 8 (B) or a whole token (C) -- each row one lane
// group, the weight and the token's table row read through L1 by every row of the block (so each
// block brings them from L2 once). A measurement device for the page's lookup-byte model, not a
// fast path: the prologue's own kernel streams chunks through a TMA ring instead.
template <typename T, typename TT, int LPR, int HS, int TS>
__global__ void rows_block_kernel(const RowArgs a, int32_t rpb) {
  constexpr int kV = HS + 2 * TS;
  const int lane = threadIdx.x & (LPR - 1);
  const int grp = threadIdx.x / LPR;
  if (grp >= rpb) return;
  const int N = a.N;
  const int hv = (N - a.R) >> 3, th = a.R >> 4, half = a.R >> 1;
  const float fN = static_cast<float>(N);
  const int32_t r = blockIdx.x * rpb + grp;
  const bool rv = r < static_cast<int32_t>(a.rows);
  const int32_t t = rv ? r / a.H : 0;
  const int32_t h = rv ? r - t * a.H : 0;
  const T* xrow = static_cast<const T*>(a.x) + (static_cast<int64_t>(t) * a.token_stride + static_cast<int64_t>(h) * N);
  uint4 xv[kV];
#pragma unroll
  for (int s = 0; s < kV; ++s)
    xv[s] = (rv && slot_ok<LPR, HS, TS>(s, lane, hv, th)) ? ld_stream16(xrow + slot_col<LPR, HS, TS>(s, lane, hv, th))
                                                         : make_uint4(0u, 0u, 0u, 0u);
  row_body<T, TT, MODE_QK, LPR, HS, TS, false>(a, r, rv, h, xv, lane, hv, th, fN, a.cos, a.sin,
                                               static_cast<int64_t>(t) * half);
}

template <typename T, typename TT>
bool launch_block_t(const RowArgs& a, int32_t rpb, cudaStream_t s) {
  const int hv = (a.N - a.R) / 8, th = a.R / 16;
  // one lane group of 8 lanes per row for head_dim <= 128 with the whole head rotated
  if (!(hv == 0 && th <= 8)) return false;
  const int threads = ((rpb * 8 + 31) / 32) * 32;
  if (threads > 1024) return false;
  const int64_t grid = (a.rows + rpb - 1) / rpb;
  if (grid > 0x7fffffffLL) return false;
  rows_block_kernel<T, TT, 8, 0, 1><<<static_cast<unsigned>(grid), threads, 0, s>>>(a, rpb);
  return true;
}

// Wide rows, RMSNorm forward: one warp per row in two passes. Pass 1 streams x (eight 16-byte
// vectors per lane in flight) for the sum of squares; pass 2 reads the row again -- it was just
// fetched, so it comes from L2, not HBM -- and writes y. Holding a 4096-wide row in registers
// would cost ~150 registers per thread and one CTA per SM; this keeps a few dozen.
template <typename T>
__global__ void __launch_bounds__(kThreads) rows_wide_fwd_kernel(const RowArgs a) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kBatch = 8;   // pass 1: vectors per lane in flight (HBM latency)
  constexpr int kBatch2 = 4;  // pass 2: the row comes back from L2
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int N = a.N;
  const int nv = N >> 3;
  const float fN = static_cast<float>(N);
  const T* w = static_cast<const T*>(a.wq);
  const int32_t rows = static_cast<int32_t>(a.rows);
  for (int32_t r = blockIdx.x * kWarps + warp; r < rows; r += gridDim.x * kWarps) {  // warp-uniform
    const T* xrow = static_cast<const T*>(a.x) + static_cast<int64_t>(r) * N;
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
    for (int v0 = lane; v0 < nv; v0 += 32 * kBatch) {
      uint4 xv[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int v = v0 + 32 * b;
        xv[b] = v < nv ? __ldg(reinterpret_cast<const uint4*>(xrow + 8 * v)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const float2 f0 = Elem<T>::unpack(xv[b].x), f1 = Elem<T>::unpack(xv[b].y);
        const float2 f2 = Elem<T>::unpack(xv[b].z), f3 = Elem<T>::unpack(xv[b].w);
        acc0 = fma2(f0, f0, acc0);
        acc1 = fma2(f1, f1, acc1);
        acc0 = fma2(f2, f2, acc0);
        acc1 = fma2(f3, f3, acc1);
      }
    }
    const float2 acc = add2(acc0, acc1);
    const float rstd = rstd_from_ss(group_sum<32>(acc.x + acc.y), fN, a.eps);
    if (a.rstd != nullptr && lane == 0) a.rstd[r] = rstd;
    const float2 rstd2 = splat2(rstd);
    T* yrow = static_cast<T*>(a.y) + static_cast<int64_t>(r) * N;
    for (int v0 = lane; v0 < nv; v0 += 32 * kBatch2) {
      uint4 xv[kBatch2], wv[kBatch2];
#pragma unroll
      for (int b = 0; b < kBatch2; ++b) {
        const int v = v0 + 32 * b;
        if (v < nv) {
          xv[b] = ld_stream16(xrow + 8 * v);
          wv[b] = ld_cached16(w + 8 * v);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch2; ++b) {
        const int v = v0 + 32 * b;
        if (v >= nv) continue;
        uint4 out;
        out.x = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(xv[b].x), rstd2), Elem<T>::unpack(wv[b].x)));
        out.y = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(xv[b].y), rstd2), Elem<T>::unpack(wv[b].y)));
        out.z = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(xv[b].z), rstd2), Elem<T>::unpack(wv[b].z)));
        out.w = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(xv[b].w), rstd2), Elem<T>::unpack(wv[b].w)));
        st_stream16(yrow + 8 * v, out);
      }
    }
  }
}

template <typename T>
bool launch_wide_fwd(const RowArgs& a, cudaStream_t s) {
  auto kern = rows_wide_fwd_kernel<T>;
  static int blocks_per_sm = -1;
  if (blocks_per_sm < 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, 0) != cudaSuccess || b < 1) b = 1;
    blocks_per_sm = b;
  }
  const int64_t need = (a.rows + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm;
  kern<<<static_cast<int>(need < cap ? need : cap), kThreads, 0, s>>>(a);
  return true;
}

// ------------------------------------------------------------------------------------------------
// Instantiation table. (LPR, HS, TS) must cover hv = (N-R)/8 <= LPR*HS and th = R/16 <= LPR*TS.
// ------------------------------------------------------------------------------------------------
struct Shape {
  int lpr, hs, ts;
};

template <typename T, typename TT, int MODE, int LPR, int HS, int TS>
bool launch_one(const RowArgs& a, cudaStream_t s) {
  // One row per lane group per iteration: two (all loads first) measured slower on the narrow-row
  // workloads (fewer CTAs, more registers); U stays a template parameter for experiments.
  constexpr int U = 1;
  auto kern = rows_vec_kernel<T, TT, MODE, LPR, HS, TS, U>;
  static int blocks_per_sm = -1;
  if (blocks_per_sm < 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, 0) != cudaSuccess || b < 1) b = 1;
    blocks_per_sm = b;
  }
  constexpr int kRowsPerCta = (kThreads / LPR) * U;
  const int64_t need = (a.rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm;
  const int grid = static_cast<int>(need < cap ? need : cap);
  size_t smem = 0;
  if (MODE == MODE_ROPE_QUANT && a.group > 0) {
    smem = static_cast<size_t>(kThreads / LPR) * (a.N / a.group) * sizeof(uint32_t);
    if (!ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem)) return false;
  }
  kern<<<grid, kThreads, smem, s>>>(a);
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
  if (MODE == MODE_FWD && a.N >= 1024) return launch_wide_fwd<T>(a, s);
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

bool launch_prologue_blocks(const RowArgs& a, int32_t rows_per_block, int dtype, int table_dtype, cudaStream_t s) {
  if (table_dtype != DT_FP32 && table_dtype != dtype) return false;
  if (dtype == DT_BF16)
    return table_dtype == DT_FP32 ? launch_block_t<__nv_bfloat16, float>(a, rows_per_block, s)
                                  : launch_block_t<__nv_bfloat16, __nv_bfloat16>(a, rows_per_block, s);
  return table_dtype == DT_FP32 ? launch_block_t<__half, float>(a, rows_per_block, s)
                                : launch_block_t<__half, __half>(a, rows_per_block, s);
}

bool launch_rows_vector(const RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s) {
  if (a.R > 0 && table_dtype != DT_FP32 && table_dtype != dtype) return false;
  if (dtype == DT_BF16) return dispatch_mode<__nv_bfloat16>(a, mode, table_dtype, s);
  if (dtype == DT_FP16) return dispatch_mode<__half>(a, mode, table_dtype, s);
  return false;
}

}  // namespace fq
