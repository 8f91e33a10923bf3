// fq_bwd.cu -- RMSNorm backward ("rmsnorm_tl.py" (Ch.17), RMSNormTileLang.backward):
//   rstd recomputed from x; xn = x*rstd; gw = g*w; c = mean(gw*xn);
//   dx = dtype(rstd*(gw - xn*c));   dw = dtype(sum over rows of g*xn).
//
// dw is a column reduction over all M rows. It is done in two deterministic stages:
//   stage 1: rows are cut into fixed chunks (a partition that depends on M only); one CTA owns a
//            chunk, computes dx for its rows and writes the chunk's fp32 partial column sums;
//   stage 2: every column adds its chunk partials in chunk order.
// No atomics anywhere, so dw is bitwise reproducible run to run and independent of the grid.
//
// Stage 1 reads x and g once and writes dx once. Rows of 1032..4096 elements take a TMA-fed kernel:
// a producer lane bulk-copies each x and g row of the chunk into a ring in shared memory, so the
// next rows are already on chip while a row is reduced (the global-load kernel, which loads two rows
// at the top of each iteration, exposes the memory latency once per iteration); eight consumer
// warps own 16-byte column vectors, hold their weights and their dw partials in registers, and meet
// once per row at a named barrier for the row's two sums. Narrower rows use 16-byte streaming loads. A row is owned by a
// team of TPR threads (a lane group for narrow rows, several warps for wide rows); one reduction
// per row yields both sum(x^2) and sum(gw*x), and c = rstd * sum(gw*x) / N (the same quantity as
// mean(gw*xn) up to fp32 rounding order).
#include "fq_device.cuh"
#include "fq_internal.h"
#include "fq_sync.cuh"

#include <cstdlib>
#include <cstring>

namespace fq {
namespace {

constexpr int kThreads = 256;
constexpr int64_t kMaxChunks = 256;

__device__ __forceinline__ uint32_t word(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

template <int TPR>
__device__ __forceinline__ float team_sum_shfl(float v) {
  return group_sum<(TPR < 32 ? TPR : 32)>(v);
}

// Two CTAs per SM (at most 128 registers) keep all <= 256 chunk CTAs resident in one wave.
template <typename T, int TPR, int VPT, int RB>
__global__ void __launch_bounds__(kThreads, 2) bwd_stage1_kernel(const BwdArgs a, int64_t rows_per_chunk) {
  constexpr int G = kThreads / TPR;               // row teams per CTA
  constexpr int WPT = TPR > 32 ? TPR / 32 : 1;    // warps per team
  __shared__ float red[2][G][WPT][2 * RB];        // cross-warp row sums (TPR > 32), double buffered
  extern __shared__ float comb[];                 // [G][VPT*TPR*8] team partials (G > 1)

  const int tid = threadIdx.x;
  const int g = tid / TPR;
  const int l = tid % TPR;
  const int N = a.N;
  const int nv = N >> 3;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * rows_per_chunk;
  const int64_t c1 = min(c0 + rows_per_chunk, a.M);
  const float fN = static_cast<float>(N);

  const T* wp = static_cast<const T*>(a.w);
  float2 wf[VPT][4];
  float2 acc[VPT][4];
  bool ok[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = l + k * TPR;
    ok[k] = v < nv;
    const uint4 u = ok[k] ? ld_cached16(wp + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      wf[k][e] = Elem<T>::unpack(word(u, e));
      acc[k][e] = make_float2(0.f, 0.f);
    }
  }

  const int64_t nrows = c1 - c0;
  const int64_t iters = (nrows + G * RB - 1) / (G * RB);
  for (int64_t it = 0; it < iters; ++it) {
    uint4 xv[RB][VPT], gv[RB][VPT];
    int64_t row[RB];
    bool rv[RB];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      row[b] = c0 + (it * RB + b) * G + g;
      rv[b] = row[b] < c1;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const bool live = rv[b] && ok[k];
        const int64_t off = row[b] * N + 8 * (l + k * TPR);
        xv[b][k] = live ? ld_stream16(static_cast<const T*>(a.x) + off) : make_uint4(0u, 0u, 0u, 0u);
        gv[b][k] = live ? ld_stream16(static_cast<const T*>(a.g) + off) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float ss[RB], sg[RB];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      float2 s2 = make_float2(0.f, 0.f), g2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 xf = Elem<T>::unpack(word(xv[b][k], e));
          const float2 gw = mul2(Elem<T>::unpack(word(gv[b][k], e)), wf[k][e]);
          s2 = fma2(xf, xf, s2);
          g2 = fma2(gw, xf, g2);
        }
      ss[b] = team_sum_shfl<TPR>(s2.x + s2.y);
      sg[b] = team_sum_shfl<TPR>(g2.x + g2.y);
    }
    if constexpr (WPT > 1) {
      const int buf = static_cast<int>(it & 1);
      const int wi = l >> 5;
      if ((l & 31) == 0) {
#pragma unroll
        for (int b = 0; b < RB; ++b) {
          red[buf][g][wi][2 * b] = ss[b];
          red[buf][g][wi][2 * b + 1] = sg[b];
        }
      }
      __syncthreads();
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        float s = 0.f, q = 0.f;
#pragma unroll
        for (int j = 0; j < WPT; ++j) {  // fixed order
          s += red[buf][g][j][2 * b];
          q += red[buf][g][j][2 * b + 1];
        }
        ss[b] = s;
        sg[b] = q;
      }
      // the other buffer is rewritten only after the next iteration's barrier
    }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      const float rstd = (a.rstd_in != nullptr) ? (rv[b] ? a.rstd_in[row[b]] : 1.f) : rstd_approx(ss[b], fN, a.eps);
      const float c = div_n(__fmul_rn(sg[b], rstd), fN);
      const float2 rstd2 = splat2(rstd), c2 = splat2(c);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        uint4 out;
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 xn = mul2(unpack_again<T>(word(xv[b][k], e)), rstd2);
          const float2 gf = unpack_again<T>(word(gv[b][k], e));
          const float2 gw = mul2(gf, wf[k][e]);
          const float2 d = sub2(gw, mul2(xn, c2));
          pk[e] = Elem<T>::pack(mul2(rstd2, d));
          acc[k][e] = fma2(gf, xn, acc[k][e]);
        }
        out = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        if (rv[b] && ok[k]) st_stream16(static_cast<T*>(a.dx) + row[b] * N + 8 * (l + k * TPR), out);
      }
    }
  }

  // Combine the G teams' column partials in team order and write this chunk's partial row.
  float* prow = a.partial + static_cast<int64_t>(blockIdx.x) * N;
  if constexpr (G == 1) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (!ok[k]) continue;
      float* p = prow + 8 * (l + k * TPR);
      reinterpret_cast<float4*>(p)[0] = make_float4(acc[k][0].x, acc[k][0].y, acc[k][1].x, acc[k][1].y);
      reinterpret_cast<float4*>(p)[1] = make_float4(acc[k][2].x, acc[k][2].y, acc[k][3].x, acc[k][3].y);
    }
  } else {
    constexpr int W = VPT * TPR * 8;  // padded row width held by one team
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 8 * (l + k * TPR) + 2 * e;
        comb[g * W + j] = acc[k][e].x;
        comb[g * W + j + 1] = acc[k][e].y;
      }
    __syncthreads();
    for (int j = tid; j < N; j += kThreads) {
      float s = 0.f;
#pragma unroll
      for (int t = 0; t < G; ++t) s += comb[t * W + j];
      prow[j] = s;
    }
  }
}

// Stage 2: dw[j] = sum over chunks of partial[chunk, j] in a fixed order. One CTA per 32 columns:
// thread (k, c4) with k in [0, 32) and c4 in [0, 8) adds chunks k, k+32, k+64, ... (in order, all
// loads in flight) for columns 4*c4..4*c4+3 of the CTA's 32; the 32 partial sums per column are
// then added in k order. The order depends on nothing but M and N: dw is reproducible bit for bit.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    bwd_stage2_kernel(const float* partial, int64_t chunks, int N, void* dw, float* dw_f32) {
  constexpr int kStreams = kThreads / 8;  // 32 chunk streams
  __shared__ float part[kStreams][33];
  // Programmatic dependent launch: this grid may be scheduled while stage 1 drains; the wait orders
  // every read of the partial sums after stage 1 has finished and its writes are visible.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int c4 = threadIdx.x & 7;
  const int k = threadIdx.x >> 3;
  const int j0 = blockIdx.x * 32 + 4 * c4;
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
  if (j0 < N) {
    const bool vec = (N % 4 == 0);
    int64_t c = k;
    for (; c + 7 * kStreams < chunks; c += 8 * kStreams) {
      float4 p[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float* src = partial + (c + u * kStreams) * N + j0;
        if (vec) {
          p[u] = *reinterpret_cast<const float4*>(src);
        } else {
          p[u].x = src[0];
          p[u].y = j0 + 1 < N ? src[1] : 0.f;
          p[u].z = j0 + 2 < N ? src[2] : 0.f;
          p[u].w = j0 + 3 < N ? src[3] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        sum.x += p[u].x;
        sum.y += p[u].y;
        sum.z += p[u].z;
        sum.w += p[u].w;
      }
    }
    for (; c < chunks; c += kStreams) {
      const float* src = partial + c * N + j0;
      sum.x += src[0];
      sum.y += j0 + 1 < N ? src[1] : 0.f;
      sum.z += j0 + 2 < N ? src[2] : 0.f;
      sum.w += j0 + 3 < N ? src[3] : 0.f;
    }
  }
  part[k][4 * c4 + 0] = sum.x;
  part[k][4 * c4 + 1] = sum.y;
  part[k][4 * c4 + 2] = sum.z;
  part[k][4 * c4 + 3] = sum.w;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int j = blockIdx.x * 32 + threadIdx.x;
    if (j < N) {
      float tot = 0.f;
#pragma unroll
      for (int q = 0; q < kStreams; ++q) tot += part[q][threadIdx.x];
      if (dw_f32) dw_f32[j] = tot;
      Elem<T>::store1(dw, j, tot);
    }
  }
}

// Scalar stage 1 for any N / alignment: one CTA per chunk walks its rows one at a time; thread i
// owns columns i, i+256, ... and accumulates its chunk partials in the workspace row.
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_stage1_scalar_kernel(const BwdArgs a, int64_t rows_per_chunk) {
  __shared__ float red[kThreads / 32][2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = a.N;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * rows_per_chunk;
  const int64_t c1 = min(c0 + rows_per_chunk, a.M);
  float* prow = a.partial + static_cast<int64_t>(blockIdx.x) * N;
  for (int j = tid; j < N; j += kThreads) prow[j] = 0.f;
  for (int64_t r = c0; r < c1; ++r) {
    float ss = 0.f, sg = 0.f;
    for (int j = tid; j < N; j += kThreads) {
      const float x = Elem<T>::load1(a.x, r * N + j);
      const float gw = __fmul_rn(Elem<T>::load1(a.g, r * N + j), Elem<T>::load1(a.w, j));
      ss = __fmaf_rn(x, x, ss);
      sg = __fmaf_rn(gw, x, sg);
    }
    ss = group_sum<32>(ss);
    sg = group_sum<32>(sg);
    if (lane == 0) {
      red[warp][0] = ss;
      red[warp][1] = sg;
    }
    __syncthreads();
    ss = 0.f;
    sg = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      ss += red[w][0];
      sg += red[w][1];
    }
    __syncthreads();
    const float rstd = (a.rstd_in != nullptr) ? a.rstd_in[r] : rstd_approx(ss, static_cast<float>(N), a.eps);
    const float c = div_n(__fmul_rn(sg, rstd), static_cast<float>(N));
    for (int j = tid; j < N; j += kThreads) {
      const float gf = Elem<T>::load1(a.g, r * N + j);
      const float xn = __fmul_rn(Elem<T>::load1(a.x, r * N + j), rstd);
      const float gw = __fmul_rn(gf, Elem<T>::load1(a.w, j));
      Elem<T>::store1(a.dx, r * N + j, __fmul_rn(rstd, __fsub_rn(gw, __fmul_rn(xn, c))));
      prow[j] = __fmaf_rn(gf, xn, prow[j]);
    }
  }
}


// ------------------------------------------------------------------------------ TMA-fed stage 1
constexpr int kStreamWarps = 8;                          // consumer warps
constexpr int kStreamThreads = (kStreamWarps + 1) * 32;  // + one producer warp

struct BwdStream {
  BwdArgs a;
  int64_t rows_per_chunk;
  unsigned int* status;
  int32_t stages;       // ring depth
  int32_t stage_bytes;  // x row + g row, multiple of 128
  int32_t depth;        // the producer keeps at most this many rows in flight
};

__host__ __device__ constexpr size_t stream_smem_bytes(int stages, int stage_bytes) {
  return 128 + static_cast<size_t>(stages) * stage_bytes + 2 * stages * sizeof(uint64_t) +
         2 * kStreamWarps * 2 * sizeof(float);
}

// Named barrier of the consumer warps that also ANDs a predicate over them: every consumer learns
// whether all of them got their data, so a failed wait never leaves the others at the barrier.
__device__ __forceinline__ bool consumers_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, 1, %2, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kStreamWarps * 32)
      : "memory");
  return r != 0;
}

// SAVED: rstd comes from the forward (a.rstd_in); the sum of squares is skipped.
template <typename T, int VPT, bool SAVED>
__global__ void __launch_bounds__(kStreamThreads, 2) bwd_stage1_stream_kernel(const BwdStream p) {
  extern __shared__ unsigned char smem_raw[];
  const BwdArgs& a = p.a;
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((128u - (raw & 127u)) & 127u);
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * p.stage_bytes);
  uint64_t* empty = full + S;
  float* red = reinterpret_cast<float*>(empty + S);  // [2][kStreamWarps][2], double buffered

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = a.N, nv = N >> 3;
  const uint32_t row_bytes = static_cast<uint32_t>(N) * sizeof(T);
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_chunk;
  const int64_t c1 = min(c0 + p.rows_per_chunk, a.M);
  const int n = static_cast<int>(c1 - c0);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStreamWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == kStreamWarps) {
    // ---------------------------------------------------------------- producer (one lane)
    if (lane != 0) return;
    int slot = 0, dslot = 0, k = 0;
    uint32_t phase = 0, dphase = 0;
    bool ok = true;
    for (; k < n; ++k) {
      if (k >= S && !mbar_wait(kWaitLimitNs, &empty[slot], phase ^ 1u)) {
        ok = false;
        break;
      }
      if (k >= p.depth) {
        if (!mbar_wait(kWaitLimitNs, &full[dslot], dphase)) {
          ok = false;
          break;
        }
        if (++dslot == S) {
          dslot = 0;
          dphase ^= 1u;
        }
      }
      unsigned char* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
      const int64_t off = (c0 + k) * static_cast<int64_t>(row_bytes);
      mbar_arrive_expect_tx(&full[slot], 2u * row_bytes);
      bulk_g2s(st, static_cast<const unsigned char*>(a.x) + off, row_bytes, &full[slot]);
      bulk_g2s(st + row_bytes, static_cast<const unsigned char*>(a.g) + off, row_bytes, &full[slot]);
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      flag_failure(p.status);
      for (int j = max(0, k - S); j < k; ++j)
        if (!mbar_wait(kWaitLimitNs, &full[j % S], static_cast<uint32_t>(j / S) & 1u)) break;
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  // Thread t owns the 16-byte column vectors t, t + 256, ...: its weights and its dw partial sums
  // stay in registers for the whole chunk.
  const T* wp = static_cast<const T*>(a.w);
  float2 wf[VPT][4], acc[VPT][4];
  bool okv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * kStreamWarps * 32;
    okv[k] = v < nv;
    const uint4 u = okv[k] ? ld_cached16(wp + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      wf[k][e] = Elem<T>::unpack(word(u, e));
      acc[k][e] = make_float2(0.f, 0.f);
    }
  }
  const float fN = static_cast<float>(N);
  int slot = 0;
  uint32_t phase = 0;
  // The saved rstd of row k is loaded one row ahead, so its global-load latency overlaps the
  // previous row's work instead of sitting between the row sums and the dx pass.
  float rstd_next = (SAVED && n > 0) ? a.rstd_in[c0] : 0.f;
  for (int k = 0; k < n; ++k) {
    const float rstd_saved = rstd_next;
    if (SAVED && k + 1 < n) rstd_next = a.rstd_in[c0 + k + 1];
    const bool got = mbar_wait(kWaitLimitNs, &full[slot], phase);
    if (!got) flag_failure(p.status);
    const unsigned char* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
    uint4 xv[VPT], gv[VPT];
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      const int v = tid + q * kStreamWarps * 32;
      const bool live = got && okv[q];
      xv[q] = live ? reinterpret_cast<const uint4*>(st)[v] : make_uint4(0u, 0u, 0u, 0u);
      gv[q] = live ? reinterpret_cast<const uint4*>(st + row_bytes)[v] : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
    if (got && lane == 0) mbar_arrive(&empty[slot]);  // the row is in registers: release the stage
    float2 s2 = make_float2(0.f, 0.f), g2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < VPT; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xf = Elem<T>::unpack(word(xv[q], e));
        const float2 gw = mul2(Elem<T>::unpack(word(gv[q], e)), wf[q][e]);
        if (!SAVED) s2 = fma2(xf, xf, s2);
        g2 = fma2(gw, xf, g2);
      }
    const float ss_w = SAVED ? 0.f : group_sum<32>(s2.x + s2.y);
    const float sg_w = group_sum<32>(g2.x + g2.y);
    float* rb = red + (k & 1) * (2 * kStreamWarps);
    if (lane == 0) {
      rb[2 * warp] = ss_w;
      rb[2 * warp + 1] = sg_w;
    }
    if (!consumers_all(got)) return;  // a stage never arrived: every consumer stops here
    // the warps' sums in fixed order, two warps per 16-byte read (rb is 16-byte aligned)
    float ss = 0.f, sg = 0.f;
#pragma unroll
    for (int w = 0; w < kStreamWarps; w += 2) {
      const float4 v = reinterpret_cast<const float4*>(rb)[w / 2];
      ss += v.x;
      sg += v.y;
      ss += v.z;
      sg += v.w;
    }
    const float rstd = SAVED ? rstd_saved : rstd_approx(ss, fN, a.eps);
    const float c = div_n(__fmul_rn(sg, rstd), fN);
    const float2 rstd2 = splat2(rstd), c2 = splat2(c);
    T* dxrow = static_cast<T*>(a.dx) + (c0 + k) * N;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xn = mul2(unpack_again<T>(word(xv[q], e)), rstd2);
        const float2 gf = unpack_again<T>(word(gv[q], e));
        const float2 d = sub2(mul2(gf, wf[q][e]), mul2(xn, c2));
        pk[e] = Elem<T>::pack(mul2(rstd2, d));
        acc[q][e] = fma2(gf, xn, acc[q][e]);
      }
      if (okv[q]) st_stream16(dxrow + 8 * (tid + q * kStreamWarps * 32), make_uint4(pk[0], pk[1], pk[2], pk[3]));
    }
    if (++slot == S) {
      slot = 0;
      phase ^= 1u;
    }
  }
  float* prow = a.partial + static_cast<int64_t>(blockIdx.x) * N;
#pragma unroll
  for (int q = 0; q < VPT; ++q) {
    if (!okv[q]) continue;
    float* pp = prow + 8 * (tid + q * kStreamWarps * 32);
    reinterpret_cast<float4*>(pp)[0] = make_float4(acc[q][0].x, acc[q][0].y, acc[q][1].x, acc[q][1].y);
    reinterpret_cast<float4*>(pp)[1] = make_float4(acc[q][2].x, acc[q][2].y, acc[q][3].x, acc[q][3].y);
  }
}

template <typename T, int VPT, bool SAVED>
bool launch_stage1_stream_t(const BwdArgs& a, const BwdPlan& plan, cudaStream_t s) {
  BwdStream p{};
  p.a = a;
  p.rows_per_chunk = plan.rows_per_chunk;
  p.status = device_status_ptr();
  p.stage_bytes = ((2 * a.N * static_cast<int>(sizeof(T))) + 127) & ~127;
  // As many stages as fit two CTAs per SM (at most 8); about 64 KB in flight per CTA.
  p.stages = static_cast<int>((110 * 1024 - stream_smem_bytes(0, 0)) / (p.stage_bytes + 16));
  if (p.stages > 8) p.stages = 8;
  if (p.stages < 2) return false;
  p.depth = (64 * 1024 + p.stage_bytes - 1) / p.stage_bytes;
  if (p.depth < 2) p.depth = 2;
  if (p.depth > p.stages) p.depth = p.stages;
  const size_t smem = stream_smem_bytes(p.stages, p.stage_bytes);
  auto kern = bwd_stage1_stream_kernel<T, VPT, SAVED>;
  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem)) return false;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.chunks));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess;
}

template <typename T, int VPT>
bool launch_stage1_stream(const BwdArgs& a, const BwdPlan& plan, cudaStream_t s) {
  return a.rstd_in != nullptr ? launch_stage1_stream_t<T, VPT, true>(a, plan, s)
                              : launch_stage1_stream_t<T, VPT, false>(a, plan, s);
}

template <typename T, int TPR, int VPT, int RB>
void launch_stage1(const BwdArgs& a, const BwdPlan& p, cudaStream_t s) {
  constexpr int G = kThreads / TPR;
  const size_t smem = (G > 1) ? static_cast<size_t>(G) * VPT * TPR * 8 * sizeof(float) : 0;
  auto kern = bwd_stage1_kernel<T, TPR, VPT, RB>;
  ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  kern<<<static_cast<unsigned>(p.chunks), kThreads, smem, s>>>(a, p.rows_per_chunk);
}

bool vector_ok(const BwdArgs& a, int dtype_size) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return (a.N % 8 == 0) && al(a.x) && al(a.w) && al(a.g) && al(a.dx) && al(a.partial) && dtype_size == 2;
}

template <typename T>
void launch_bwd_t(const BwdArgs& a, cudaStream_t s) {
  const BwdPlan p = bwd_plan(a.M);
  if (a.M > 0) {
    const int nv = a.N / 8;
    const bool vec = vector_ok(a, sizeof(T));
    const char* sel = getenv("FQ_BWD_KERNEL");  // "generic": the global-load kernel (diagnostic switch)
    const bool stream = vec && nv > 128 && nv <= 512 && !(sel != nullptr && strcmp(sel, "generic") == 0);
    if (stream && nv <= 256 && launch_stage1_stream<T, 1>(a, p, s)) {
    } else if (stream && launch_stage1_stream<T, 2>(a, p, s)) {
    } else if (vec && nv <= 16) launch_stage1<T, 16, 1, 2>(a, p, s);
    else if (vec && nv <= 32) launch_stage1<T, 32, 1, 2>(a, p, s);
    else if (vec && nv <= 64) launch_stage1<T, 64, 1, 2>(a, p, s);
    else if (vec && nv <= 128) launch_stage1<T, 128, 1, 2>(a, p, s);
    else if (vec && nv <= 256) launch_stage1<T, 256, 1, 2>(a, p, s);
    else if (vec && nv <= 512) launch_stage1<T, 256, 2, 2>(a, p, s);
    else if (vec && nv <= 1024) launch_stage1<T, 256, 4, 1>(a, p, s);
    else bwd_stage1_scalar_kernel<T><<<static_cast<unsigned>(p.chunks), kThreads, 0, s>>>(a, p.rows_per_chunk);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>((a.N + 31) / 32));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, bwd_stage2_kernel<T>, static_cast<const float*>(a.partial), p.chunks, a.N, a.dw, a.dw_f32);
}

}  // namespace

BwdPlan bwd_plan(int64_t M) {
  BwdPlan p;
  if (M <= 0) {
    p.chunks = 0;
    p.rows_per_chunk = 1;
    return p;
  }
  p.rows_per_chunk = (M + kMaxChunks - 1) / kMaxChunks;
  p.chunks = (M + p.rows_per_chunk - 1) / p.rows_per_chunk;
  return p;
}

size_t bwd_workspace_bytes(int64_t M, int64_t N) {
  const BwdPlan p = bwd_plan(M);
  return static_cast<size_t>(p.chunks) * static_cast<size_t>(N) * sizeof(float);
}

void launch_bwd(const BwdArgs& a, int dtype, cudaStream_t s) {
  if (dtype == DT_BF16) launch_bwd_t<__nv_bfloat16>(a, s);
  else launch_bwd_t<__half>(a, s);
}

}  // namespace fq
