// fq_rows_tma.cu -- TMA-fed persistent kernels for RMSNorm forward, RMSNorm + NeoX partial RoPE
// (+ FP8) and LayerNorm forward over contiguous rows ("rmsnorm_tl.py" (Ch.17), _rmsnorm_fwd;
// "rmsnorm_rope_quant.py" (Ch.13 fusion), rms_norm_rope_fused / rms_norm_rope_quant_fused /
// torch_reference_fused; "ledger.py" (Ch.13 ledger), layer_norm).
//
// The rows are cut into stages of SR consecutive rows, one per CTA of the grid. The CTAs that are
// resident take over the stages of CTAs that have not started yet through cluster launch control (a
// hardware work queue: no counter in global memory), so every SM keeps streaming until the last
// stage is taken. One producer lane streams its stages through a ring in shared memory with
// cp.async.bulk: a stage is SR consecutive x rows (one bulk copy) and, with rotation, their SR cos
// and SR sin table rows (the tables of these calls have one row per x row); an mbarrier counts the
// bytes and every wait is bounded (fq_sync.cuh). Bytes in flight do not depend on registers, which is
// what the register-hungry, latency-bound global-load kernels lacked. The consumer warps read x from
// the stage:
//   - narrow rows: eight consumer warps with the lane-group layout and arithmetic of the generic row
//     kernel (fq_rows.cuh), one row per lane group per stage, tables read from the stage; the warps
//     work as one group or as several groups that take the stages in turn (finer work units);
//   - wide rows, shared memory (RMSNorm forward beyond 4096 columns, RMSNorm + RoPE, the quantising
//     shapes the register kernels do not take): four consumer warps, one row per warp per stage,
//     two or three passes over the staged row; the weight row is copied into shared memory once per
//     CTA. Two CTAs share an SM, so a stage is four rows and the ring fills and drains in small steps;
//   - wide rows, registers (RMSNorm forward, RMSNorm + RoPE + FP8 and LayerNorm on rows of 1024 to
//     4096): one CTA per SM, two, three or five consumer groups of four warps taking the stages in
//     turn, one or two warps per row; a warp copies its row into registers and releases the stage
//     at once.
// y is written with 16-byte evict-first stores. x and the tables are read from HBM exactly once.
#include <cstdlib>
#include <string>
#include <type_traits>

#include "fq_device.cuh"
#include "fq_internal.h"
#include "fq_rows.cuh"
#include "fq_sync.cuh"

namespace fq {
namespace {

using namespace rows;

constexpr int kConsumerWarps = 8;  // narrow-row kernel
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kWideWarps = 4;  // wide-row kernel
constexpr int kWideThreads = (kWideWarps + 1) * 32;
constexpr int kWideUnroll = 4;

struct StreamArgs {
  RowArgs a;
  unsigned int* status;
  int32_t stages;       // ring depth
  int32_t stage_bytes;  // x block + 2 table blocks, multiple of 128
  int32_t tab_off;      // byte offset of the cos block in a stage (0 when there is no rotation)
  int32_t tab_block;    // bytes of one table block
  int32_t depth;        // the producer keeps at most this many stages in flight
  int32_t w_bytes;      // bytes of the weight row staged once per CTA (0: none)
  int32_t b_bytes;      // bytes of a second row (the LayerNorm bias) staged right after it (0: none)
};

constexpr int kReq = 2;  // cluster-launch-control requests a producer keeps in flight

// Producer: one lane streams the stages this CTA takes (its own first, then those of CTAs it takes
// over), posts `markers` end markers (one per group of consumer warps that take stages in turn), and
// returns. Its first kReq work requests were started before the dependency wait (ring_setup).
__device__ __forceinline__ void produce(const StreamArgs& p, unsigned char* smem, uint64_t* full, uint64_t* empty,
                                        uint64_t* wbar, unsigned char* wsm, uint4* resp, uint64_t* cbar,
                                        int32_t* stage_row, int SR, int esize, int tsize, int markers = 1) {
  const RowArgs& a = p.a;
  const int S = p.stages;
  if (p.w_bytes > 0) {
    mbar_arrive_expect_tx(wbar, static_cast<uint32_t>(p.w_bytes + p.b_bytes));
    bulk_g2s(wsm, a.wq, static_cast<uint32_t>(p.w_bytes), wbar);
    if (p.b_bytes > 0) bulk_g2s(wsm + p.w_bytes, a.bias, static_cast<uint32_t>(p.b_bytes), wbar);
  }
  const uint32_t xrow = static_cast<uint32_t>(a.N) * esize;
  const uint32_t trow = static_cast<uint32_t>(a.R / 2) * tsize;
  int slot = 0, dslot = 0;
  uint32_t phase = 0, dphase = 0;
  int k = 0;
  bool ok = true;
  // The kReq first work requests were issued by ring_setup.
  ClcQueue<kReq> queue{resp, cbar, kReq, 0, false};
  uint32_t chunk = blockIdx.x;
  for (;;) {
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
    const int32_t rs = static_cast<int32_t>(chunk) * SR;
    const uint32_t nr = static_cast<uint32_t>(min(SR, static_cast<int32_t>(a.rows) - rs));
    unsigned char* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
    const uint32_t tb = (a.R > 0) ? nr * trow : 0u;
    stage_row[slot] = rs;  // published to the consumers by the barrier's phase completion
    mbar_arrive_expect_tx(&full[slot], nr * xrow + 2u * tb);
    bulk_g2s(st, static_cast<const unsigned char*>(a.x) + static_cast<int64_t>(rs) * xrow, nr * xrow, &full[slot]);
    if (tb > 0) {
      bulk_g2s(st + p.tab_off, static_cast<const unsigned char*>(a.cos) + static_cast<int64_t>(rs) * trow, tb,
               &full[slot]);
      bulk_g2s(st + p.tab_off + p.tab_block,
               static_cast<const unsigned char*>(a.sin) + static_cast<int64_t>(rs) * trow, tb, &full[slot]);
    }
    ++k;
    if (++slot == S) {
      slot = 0;
      phase ^= 1u;
    }
    // The next stage: a chunk taken over from a CTA that has not started (none left: done).
    const int got = queue.next(&chunk);
    if (got < 0) ok = false;
    if (got <= 0) break;
  }
  // End markers: one stage each, so that every group of consumer warps meets one.
  for (int e = 0; ok && e < markers; ++e) {
    if (k >= S && !mbar_wait(kWaitLimitNs, &empty[slot], phase ^ 1u)) {
      ok = false;
      break;
    }
    stage_row[slot] = -1;
    mbar_arrive(&full[slot]);
    ++k;
    if (++slot == S) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (ok) return;
  flag_failure(p.status);
  for (int j = max(0, k - S); j < k; ++j)
    if (!mbar_wait(kWaitLimitNs, &full[j % S], static_cast<uint32_t>(j / S) & 1u)) break;
  queue.drain();
}

// Shared set-up of both kernels: ring layout, barriers, programmatic-launch handshake, the first
// work requests.
// Shared memory: [pad to 128][stages x stage_bytes][kReq x 16-byte responses][full x stages]
// [empty x stages][request barriers x kReq][wbar][stage start rows x stages][pad to 128][weight row].
struct Ring {
  unsigned char* smem;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* wbar;
  unsigned char* w;
  uint4* resp;
  uint64_t* cbar;
  int32_t* stage_row;
};

__host__ __device__ constexpr size_t ring_bytes(int stages, int stage_bytes, int w_bytes) {
  return 128 + static_cast<size_t>(stages) * stage_bytes + kReq * 16 + (2 * stages + kReq + 1) * sizeof(uint64_t) +
         stages * sizeof(int32_t) + 128 + w_bytes;
}

// `consumers`: warps that release each stage; the producer is warp `producer_warp` (default: the
// warp after `consumers`).
__device__ __forceinline__ Ring ring_setup(const StreamArgs& p, unsigned char* smem_raw, int consumers,
                                           int producer_warp = -1) {
  Ring g;
  const uint32_t raw = smem_addr(smem_raw);
  g.smem = smem_raw + ((128u - (raw & 127u)) & 127u);
  g.resp = reinterpret_cast<uint4*>(g.smem + static_cast<size_t>(p.stages) * p.stage_bytes);
  g.full = reinterpret_cast<uint64_t*>(g.resp + kReq);
  g.empty = g.full + p.stages;
  g.cbar = g.empty + p.stages;
  g.wbar = g.cbar + kReq;
  g.stage_row = reinterpret_cast<int32_t*>(g.wbar + 1);
  const uintptr_t wend = reinterpret_cast<uintptr_t>(g.stage_row + p.stages);
  g.w = reinterpret_cast<unsigned char*>((wend + 127) & ~static_cast<uintptr_t>(127));
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&g.full[s], 1);
      mbar_init(&g.empty[s], consumers);
    }
    for (int c = 0; c < kReq; ++c) mbar_init(&g.cbar[c], 1);
    mbar_init(g.wbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The work requests touch no data of the previous kernel: the producer lane starts them before the
  // dependency wait. Every global access comes after it.
  if (threadIdx.x == (producer_warp < 0 ? consumers : producer_warp) * 32)
    for (int c = 0; c < kReq; ++c) clc_try_cancel(&g.resp[c], &g.cbar[c]);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  return g;
}

// ---------------------------------------------------------------------------------- narrow rows
// Up to four vectors per lane (and the four-lane fp16 rotary shape) the kernel fits two CTAs per SM
// without spilling; wider rows take one. G consumer groups take the stages in turn (stage k goes to
// group k % G): a stage holds 1/G of the rows, so a launch has G times as many work units to spread
// over the SMs.
template <typename T, typename TT, int MODE, int LPR, int HS, int TS, int G = 1>
__global__ void __launch_bounds__(kThreads, ((HS + 2 * TS) <= 4 || LPR <= 4) ? 2 : 1) rows_tma_kernel(const StreamArgs p) {
  extern __shared__ unsigned char smem_raw[];
  constexpr int kV = HS + 2 * TS;
  constexpr int kGroupWarps = kConsumerWarps / G;
  constexpr int SR = kGroupWarps * (32 / LPR);  // one row per lane group per stage
  const Ring g = ring_setup(p, smem_raw, kGroupWarps, kConsumerWarps);
  const RowArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane32 = threadIdx.x & 31;
  if (warp == kConsumerWarps) {
    if (lane32 == 0)
      produce(p, g.smem, g.full, g.empty, g.wbar, g.w, g.resp, g.cbar, g.stage_row, SR, sizeof(T), sizeof(TT), G);
    return;
  }
  const int lane = lane32 & (LPR - 1);
  const int l = (warp % kGroupWarps) * (32 / LPR) + lane32 / LPR;  // row within each stage
  const int N = a.N;
  const int hv = (N - a.R) >> 3, th = a.R >> 4, half = a.R >> 1;
  const float fN = static_cast<float>(N);
  // This lane's weight vectors are the same for every row: load them once.
  uint4 wv[kV];
  const T* w = static_cast<const T*>(a.wq);
#pragma unroll
  for (int s = 0; s < kV; ++s)
    wv[s] = slot_ok<LPR, HS, TS>(s, lane, hv, th) ? ld_cached16(w + slot_col<LPR, HS, TS>(s, lane, hv, th))
                                                  : make_uint4(0u, 0u, 0u, 0u);
  int slot = warp / kGroupWarps;  // this group's first stage; it takes every G-th after it
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait(kWaitLimitNs, &g.full[slot], phase)) {
      flag_failure(p.status);
      return;
    }
    const int32_t rs = g.stage_row[slot];
    if (rs < 0) break;  // end marker
    const unsigned char* st = g.smem + static_cast<size_t>(slot) * p.stage_bytes;
    const bool live = l < static_cast<int32_t>(a.rows) - rs;
    const int lr = live ? l : 0;  // dead lane groups read row 0 of the stage (always present)
    const T* xs = reinterpret_cast<const T*>(st) + static_cast<int64_t>(lr) * N;
    uint4 xv[kV];
#pragma unroll
    for (int s = 0; s < kV; ++s)
      xv[s] = slot_ok<LPR, HS, TS>(s, lane, hv, th)
                  ? *reinterpret_cast<const uint4*>(xs + slot_col<LPR, HS, TS>(s, lane, hv, th))
                  : make_uint4(0u, 0u, 0u, 0u);
    row_body<T, TT, MODE, LPR, HS, TS, true, true>(a, rs + l, live, 0, xv, lane, hv, th, fN, st + p.tab_off,
                                                    st + p.tab_off + p.tab_block, static_cast<int64_t>(lr) * half, wv);
    __syncwarp();
    if (lane32 == 0) mbar_arrive(&g.empty[slot]);  // x and this stage's table rows have been read
    slot += G;  // the ring holds a multiple of G stages: a slot always belongs to the same group
    if (slot >= p.stages) {
      slot -= p.stages;
      phase ^= 1u;
    }
  }
}

// ---------------------------------------------------------------------------------- wide rows
template <typename T>
__device__ __forceinline__ float2 sq_acc(uint4 u, float2 acc) {
  const float2 f0 = Elem<T>::unpack(u.x), f1 = Elem<T>::unpack(u.y);
  const float2 f2 = Elem<T>::unpack(u.z), f3 = Elem<T>::unpack(u.w);
  acc = fma2(f0, f0, acc);
  acc = fma2(f1, f1, acc);
  acc = fma2(f2, f2, acc);
  return fma2(f3, f3, acc);
}

// The same sums with the squares taken straight from the 16-bit operands (fma.rn.f32.bf16 / .f16):
// x^2 of a 16-bit value is exact in fp32 and each step rounds once, as fma2 on the unpacked values
// does, so the sums are bit-identical without unpacking x (fewer instructions and registers: the
// register-resident kernels below no longer spill and fit one more consumer group).
template <typename T>
__device__ __forceinline__ float2 sq_acc_mixed(uint4 u, float2 acc) {
  acc = Mixed<T>::sq_add(u.x, acc);
  acc = Mixed<T>::sq_add(u.y, acc);
  acc = Mixed<T>::sq_add(u.z, acc);
  return Mixed<T>::sq_add(u.w, acc);
}

template <typename T>
__device__ __forceinline__ uint4 norm8(uint4 u, uint4 wv, float2 rstd2) {
  uint4 out;
  out.x = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(u.x), rstd2), Elem<T>::unpack(wv.x)));
  out.y = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(u.y), rstd2), Elem<T>::unpack(wv.y)));
  out.z = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(u.z), rstd2), Elem<T>::unpack(wv.z)));
  out.w = Elem<T>::pack(mul2(mul2(Elem<T>::unpack(u.w), rstd2), Elem<T>::unpack(wv.w)));
  return out;
}

template <typename T>
__global__ void __launch_bounds__(kWideThreads) rows_tma_wide_fwd_kernel(const StreamArgs p) {
  extern __shared__ unsigned char smem_raw[];
  constexpr int SR = kWideWarps;  // one row per warp per stage
  constexpr int U = kWideUnroll;
  static_assert(U == 4, "the partial sums below are combined for four accumulators");
  const Ring g = ring_setup(p, smem_raw, kWideWarps);
  const RowArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kWideWarps) {
    if (lane == 0) produce(p, g.smem, g.full, g.empty, g.wbar, g.w, g.resp, g.cbar, g.stage_row, SR, sizeof(T), 2);
    return;
  }
  const int N = a.N, nv = N >> 3;
  const float fN = static_cast<float>(N);
  const uint4* ws = reinterpret_cast<const uint4*>(g.w);
  if (!mbar_wait(kWaitLimitNs, g.wbar, 0u)) {
    flag_failure(p.status);
    return;
  }
  int slot = 0;
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait(kWaitLimitNs, &g.full[slot], phase)) {
      flag_failure(p.status);
      return;
    }
    const int32_t rs = g.stage_row[slot];
    if (rs < 0) break;  // end marker
    const int32_t r = rs + warp;
    if (r < static_cast<int32_t>(a.rows)) {  // warp-uniform
      const uint4* xs = reinterpret_cast<const uint4*>(g.smem + static_cast<size_t>(slot) * p.stage_bytes +
                                                       static_cast<size_t>(warp) * N * sizeof(T));
      float2 acc[U];
#pragma unroll
      for (int j = 0; j < U; ++j) acc[j] = make_float2(0.f, 0.f);
      int v = lane;
      for (; v + 32 * (U - 1) < nv; v += 32 * U) {
        uint4 u[U];
#pragma unroll
        for (int j = 0; j < U; ++j) u[j] = xs[v + 32 * j];
#pragma unroll
        for (int j = 0; j < U; ++j) acc[j] = sq_acc<T>(u[j], acc[j]);
      }
      for (; v < nv; v += 32) acc[0] = sq_acc<T>(xs[v], acc[0]);
      const float2 s01 = add2(acc[0], acc[1]), s23 = add2(acc[2], acc[3]);
      const float2 sum = add2(s01, s23);
      const float rstd = rstd_from_ss(group_sum<32>(sum.x + sum.y), fN, a.eps);
      if (a.rstd != nullptr && lane == 0) a.rstd[r] = rstd;
      const float2 rstd2 = splat2(rstd);
      uint4* yrow = reinterpret_cast<uint4*>(static_cast<T*>(a.y) + static_cast<int64_t>(r) * N);
      v = lane;
      for (; v + 32 * (U - 1) < nv; v += 32 * U) {
        uint4 u[U], wv[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          u[j] = xs[v + 32 * j];
          wv[j] = ws[v + 32 * j];
        }
#pragma unroll
        for (int j = 0; j < U; ++j) st_stream16(yrow + v + 32 * j, norm8<T>(u[j], wv[j], rstd2));
      }
      for (; v < nv; v += 32) st_stream16(yrow + v, norm8<T>(xs[v], ws[v], rstd2));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[slot]);
    if (++slot == p.stages) {
      slot = 0;
      phase ^= 1u;
    }
  }
}

// ------------------------------------------------------------------ wide rows, rotation (+ FP8)
// RMSNorm + NeoX partial RoPE, and with QUANT the per-row or group-wise FP8 codes, for rows of
// N >= 1024: four consumer warps, one row per warp per stage. Pass 1: sum of squares over the
// staged row. Pass 2: head vectors normalised, rotary pairs normalised and rotated (both members of
// a pair and the row's cos/sin entries are in shared memory: no shuffle), each result rounded to
// the storage dtype as the definition does, written to y and -- when quantising -- back into the
// row's own place in the stage. Pass 3 (QUANT): codes from the staged y with the row's (or the
// group's) scale. Group maxima: atomicMax on the float bits in a per-warp array of N / group words.
template <typename T, typename TT, bool QUANT>
__global__ void __launch_bounds__(kWideThreads) rows_tma_wide_rope_kernel(const StreamArgs p) {
  extern __shared__ unsigned char smem_raw[];
  constexpr int SR = kWideWarps;  // one row per warp per stage
  const Ring g = ring_setup(p, smem_raw, kWideWarps);
  const RowArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kWideWarps) {
    if (lane == 0)
      produce(p, g.smem, g.full, g.empty, g.wbar, g.w, g.resp, g.cbar, g.stage_row, SR, sizeof(T), sizeof(TT));
    return;
  }
  const int N = a.N, nv = N >> 3, hv = (N - a.R) >> 3, th = a.R >> 4, half = a.R >> 1;
  const float fN = static_cast<float>(N);
  const uint4* ws = reinterpret_cast<const uint4*>(g.w);
  const bool grouped = QUANT && a.group > 0;
  const int gs = grouped ? a.group : N;
  const int G = N / gs;
  // Per warp: [G] group maxima (float bits), then [G] scales and [G] reciprocals.
  uint32_t* gmax = grouped ? reinterpret_cast<uint32_t*>(g.w + p.w_bytes) + warp * 3 * G : nullptr;
  float* gsc = grouped ? reinterpret_cast<float*>(gmax + G) : nullptr;
  float* grc = grouped ? gsc + G : nullptr;
  const bool clamp = a.fp8_max != 448.0f;
  if (!mbar_wait(kWaitLimitNs, g.wbar, 0u)) {
    flag_failure(p.status);
    return;
  }
  int slot = 0;
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait(kWaitLimitNs, &g.full[slot], phase)) {
      flag_failure(p.status);
      return;
    }
    const int32_t rs = g.stage_row[slot];
    if (rs < 0) break;  // end marker
    const int32_t r = rs + warp;
    if (r < static_cast<int32_t>(a.rows)) {  // warp-uniform
      unsigned char* st = g.smem + static_cast<size_t>(slot) * p.stage_bytes;
      uint4* xs = reinterpret_cast<uint4*>(st + static_cast<size_t>(warp) * N * sizeof(T));
      const TT* cs = reinterpret_cast<const TT*>(st + p.tab_off) + warp * half;
      const TT* sn = reinterpret_cast<const TT*>(st + p.tab_off + p.tab_block) + warp * half;
      // pass 1: sum of squares
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      for (int v = lane; v < nv; v += 32) {
        const uint4 u = xs[v];
        const float2 f0 = Elem<T>::unpack(u.x), f1 = Elem<T>::unpack(u.y);
        const float2 f2 = Elem<T>::unpack(u.z), f3 = Elem<T>::unpack(u.w);
        acc0 = fma2(f0, f0, acc0);
        acc1 = fma2(f1, f1, acc1);
        acc0 = fma2(f2, f2, acc0);
        acc1 = fma2(f3, f3, acc1);
      }
      const float2 acc = add2(acc0, acc1);
      const float ssr = group_sum<32>(acc.x + acc.y);
      const float2 rstd2 = splat2(QUANT ? rstd_from_ss(ssr, fN, a.eps) : rstd_approx(ssr, fN, a.eps));
      T* yrow = a.y != nullptr ? static_cast<T*>(a.y) + static_cast<int64_t>(r) * N : nullptr;
      float amax = 0.f;
      if (grouped) {
        __syncwarp();  // the previous row's readers of the group maxima are done
        for (int q = lane; q < G; q += 32) gmax[q] = 0u;
        __syncwarp();
      }
      // pass 2a: head columns
      for (int v = lane; v < hv; v += 32) {
        const uint4 u = xs[v], wv = ws[v];
        uint4 out;
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t pk =
              Elem<T>::pack(mul2(mul2(Elem<T>::unpack(rows::word(u, k)), rstd2), Elem<T>::unpack(rows::word(wv, k))));
          rows::set_word(out, k, pk);
          if (QUANT) {
            const float2 rn = Elem<T>::unpack(pk);
            m = fmaxf(m, fmaxf(fabsf(rn.x), fabsf(rn.y)));
          }
        }
        if (yrow != nullptr) st_stream16(yrow + 8 * v, out);
        if (QUANT) {
          xs[v] = out;
          amax = fmaxf(amax, m);
          if (grouped) atomicMax(&gmax[(8 * v) / gs], __float_as_uint(m));
        }
      }
      // pass 2b: rotary pairs (tail-lo vector hv + i with tail-hi vector hv + th + i)
      for (int i = lane; i < th; i += 32) {
        const int vlo = hv + i, vhi = hv + th + i;
        const uint4 ulo = xs[vlo], uhi = xs[vhi], wlo = ws[vlo], whi = ws[vhi];
        float2 c[4], s4[4];
        rows::load_table8<TT, true>(cs, 8 * i, c);
        rows::load_table8<TT, true>(sn, 8 * i, s4);
        uint4 plo4, phi4;
        float mlo = 0.f, mhi = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 lo =
              round_trip<T>(mul2(mul2(Elem<T>::unpack(rows::word(ulo, k)), rstd2), Elem<T>::unpack(rows::word(wlo, k))));
          const float2 hi =
              round_trip<T>(mul2(mul2(Elem<T>::unpack(rows::word(uhi, k)), rstd2), Elem<T>::unpack(rows::word(whi, k))));
          const uint32_t plo = Elem<T>::pack(sub2(mul2(lo, c[k]), mul2(hi, s4[k])));
          const uint32_t phi = Elem<T>::pack(add2(mul2(hi, c[k]), mul2(lo, s4[k])));
          rows::set_word(plo4, k, plo);
          rows::set_word(phi4, k, phi);
          if (QUANT) {
            const float2 rl = Elem<T>::unpack(plo), rh = Elem<T>::unpack(phi);
            mlo = fmaxf(mlo, fmaxf(fabsf(rl.x), fabsf(rl.y)));
            mhi = fmaxf(mhi, fmaxf(fabsf(rh.x), fabsf(rh.y)));
          }
        }
        if (yrow != nullptr) {
          st_stream16(yrow + 8 * vlo, plo4);
          st_stream16(yrow + 8 * vhi, phi4);
        }
        if (QUANT) {
          xs[vlo] = plo4;
          xs[vhi] = phi4;
          amax = fmaxf(amax, fmaxf(mlo, mhi));
          if (grouped) {
            atomicMax(&gmax[(8 * vlo) / gs], __float_as_uint(mlo));
            atomicMax(&gmax[(8 * vhi) / gs], __float_as_uint(mhi));
          }
        }
      }
      if constexpr (QUANT) {
        // pass 3: codes from the staged y
        __syncwarp();
        const float sc = __fdiv_rn(fmaxf(group_max<32>(amax), 1e-4f), a.fp8_max);
        const float rc = __frcp_rn(sc);
        if (grouped) {  // one scale and reciprocal per group, then written out
          for (int q = lane; q < G; q += 32) {
            const float sg = __fdiv_rn(fmaxf(__uint_as_float(gmax[q]), 1e-4f), a.fp8_max);
            gsc[q] = sg;
            grc[q] = __frcp_rn(sg);
            a.scale[static_cast<int64_t>(r) * G + q] = sg;
          }
          __syncwarp();
        }
        uint8_t* qrow = a.q + static_cast<int64_t>(r) * N;
        for (int v = lane; v < nv; v += 32) {
          const uint4 u = xs[v];
          float s_v = sc, r_v = rc;
          if (grouped) {
            const int q = (8 * v) / gs;
            s_v = gsc[q];
            r_v = grc[q];
          }
          float2 q4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            q4[k] = div2_by(Elem<T>::unpack(rows::word(u, k)), s_v, r_v);
            if (clamp) q4[k] = make_float2(clamp_abs(q4[k].x, a.fp8_max), clamp_abs(q4[k].y, a.fp8_max));
          }
          st_stream8(qrow + 8 * v, pack_e4m3x8(q4[0], q4[1], q4[2], q4[3]));
        }
        if (!grouped && lane == 0) a.scale[r] = sc;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[slot]);
    if (++slot == p.stages) {
      slot = 0;
      phase ^= 1u;
    }
  }
}

// ------------------------------------------------------- wide rows, FP8, register-resident rows
// RMSNorm + NeoX partial RoPE + FP8 codes with one scale per row or per group of columns
// ("rmsnorm_rope_quant.py" (Ch.13 fusion), rms_norm_rope_quant_fused) for rows of N = 256 * VPT
// elements, rope_dim <= 256, group sizes that are powers of two. Consumer warps in groups of four
// take the stages in turn (one CTA per SM; the ring holds a multiple of the group count); each warp copies its row -- VPT 16-byte vectors per lane, vector v = lane + 32k --
// into registers, and with it, on the lanes that hold rotary vectors (all in the last slot, since
// N / 8 is a multiple of 32 and rope_dim / 8 <= 32), the rotation partner's vector and the eight
// cos and sin entries of its pairs; then it releases the stage. Everything after that runs on
// registers: the sum of squares; y = dtype(x * rstd * w) per vector, the rotary lanes rotating
// their own and their partner's normalised values (each lane computes its own output: lo' = lo*c -
// hi*s on the lo side, hi' = hi*c + lo*s on the hi side, the same rounded operations as the
// definition); the |y| maxima (per row over the warp; per group over the group's lanes of a slot,
// then across slots for groups of more than 32 vectors); and the codes as correctly rounded
// quotients. The warp's rows and the stage ring are independent, so the copy of the next stages
// overlaps this work.
// Warps per consumer group (a stage holds kRegRows / TPR rows). Consumer groups take the stages in
// turn: five when a warp holds up to 8 vector slots (21 warps, 80 registers per thread), three for
// 12 slots (13 warps: registers are allotted for 16, so 128 per thread), two for 16 slots, whose 64
// registers of row data need more room (168 per thread). Rows of 4096 are split over two warps of 8
// slots each, so they run with five groups: ten rows in flight per SM. The kernels are latency-bound,
// so rows in flight count most; measured on the 4096 x 4096 workloads (RMSNorm + RoPE + FP8,
// LayerNorm) and the 8192 x 4096 RMSNorm forward, in us: three groups 11.79, 12.11, 21.48; four
// 10.82 (after the mixed-precision squares, which removed a spill), 11.76, 21.28; five 10.66, 11.55,
// 21.19; six (72 registers) 10.76, 11.54, 21.19.
constexpr int kRegRows = 4;
__host__ __device__ constexpr int reg_groups(int vpt) { return vpt <= 8 ? 5 : (vpt <= 12 ? 3 : 2); }
__host__ __device__ constexpr int reg_threads(int groups) { return (kRegRows * groups + 1) * 32; }

// RN(m / fmax) from rcp = RN(1 / fmax): one product and Markstein's correction (the residual
// m - s0 * fmax is exact in one FMA). m >= 1e-4 and fmax a normal float keep every step normal.
__device__ __forceinline__ float scale_of(float m, float fmax, float rcp) {
  const float s0 = __fmul_rn(m, rcp);
  return __fmaf_rn(__fmaf_rn(-s0, fmax, m), rcp, s0);
}

// Reduce-scatter of per-slot maxima over segments of SEG lanes (VPT values per lane, both powers of
// two): at each level the lanes of a pair (lane mask O) keep opposite halves of their values and take
// the maximum with the partner's copy of the half they keep; once a lane is down to one value the
// remaining levels are plain max-reductions. Afterwards lane j of a segment holds in m[i]
// (i < max(1, VPT / SEG)) the segment's maximum of slot i + floor(j * VPT / SEG).
template <int N, int O, int VPT>
__device__ __forceinline__ void seg_reduce_scatter(float (&m)[VPT], int lane) {
  const bool upper = (lane & O) != 0;
  if constexpr (N > 1) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float keep = upper ? m[i + N / 2] : m[i];
      const float send = upper ? m[i] : m[i + N / 2];
      m[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, O));
    }
  } else {
    m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], O));
  }
  if constexpr (O > 1) seg_reduce_scatter<(N > 1 ? N / 2 : 1), O / 2, VPT>(m, lane);
}

// norm8 that also folds the fp32 values' |v| maximum into m before they are rounded to the storage
// dtype. Rounding to nearest is monotone and odd, so max_i |RN(v_i)| = RN(max_i |v_i|): the maximum
// of the rounded y is the rounded maximum, taken without unpacking y again.
template <typename T>
__device__ __forceinline__ uint4 norm8_max(uint4 u, uint4 wv, float2 rstd2, float& m) {
  const float2 v0 = mul2(mul2(Elem<T>::unpack(u.x), rstd2), Elem<T>::unpack(wv.x));
  const float2 v1 = mul2(mul2(Elem<T>::unpack(u.y), rstd2), Elem<T>::unpack(wv.y));
  const float2 v2 = mul2(mul2(Elem<T>::unpack(u.z), rstd2), Elem<T>::unpack(wv.z));
  const float2 v3 = mul2(mul2(Elem<T>::unpack(u.w), rstd2), Elem<T>::unpack(wv.w));
  m = absmax4(absmax4(m, v0, v1), v2, v3);
  return make_uint4(Elem<T>::pack(v0), Elem<T>::pack(v1), Elem<T>::pack(v2), Elem<T>::pack(v3));
}

// Maximum of v over the warp in one instruction (redux.sync on f32, sm_100-class SMs) instead of five
// shuffle-and-max levels. A maximum selects one of its inputs, so the result equals the shuffle
// tree's for the non-negative, non-NaN |y| maxima it is used on.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// The storage dtype's rounding of one fp32 value, as fp32.
template <typename T>
__device__ __forceinline__ float round_to(float m) {
  return Elem<T>::unpack(Elem<T>::pack(make_float2(m, m))).x;
}

// Codes of eight stored y values as e4m3(RN(y * r)), r = RN(1 / scale): within one fp32 ulp of the
// quotient y / scale, so a code can differ from the quotient's only where y / scale sits at an e4m3
// rounding boundary. The product keeps the sign of zero (y = -0 codes as 0x80, as y / scale does).
template <typename T>
__device__ __forceinline__ uint2 codes8_rcp(uint4 y, float r, bool clamp, float fmax) {
  float2 q[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    q[e] = mul2(Elem<T>::unpack(rows::word(y, e)), splat2(r));
    if (clamp) q[e] = make_float2(clamp_abs(q[e].x, fmax), clamp_abs(q[e].y, fmax));
  }
  return pack_e4m3x8(q[0], q[1], q[2], q[3]);
}

// Barrier of the TPR warps that share a row (named barrier 1 + team); team_all also ANDs a predicate
// over them, so a failed wait in one warp stops its partner at the same point instead of leaving it
// at a later barrier.
__device__ __forceinline__ void team_sync(int team, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(threads) : "memory");
}

__device__ __forceinline__ bool team_all(bool v, int team, int threads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(1 + team), "r"(threads)
      : "memory");
  return r != 0;
}

// GV: 0 = one scale per row; > 0 = groups of GV vectors (8 * GV columns, GV <= 32) reduced by a
// reduce-scatter; -1 = any power-of-two group size, reduced per slot.
// TPR: warps per row. With two, each warp holds one contiguous half of the row (VPT / 2 slots), the
// pair adds its sums of squares and takes the larger |y| maximum through shared memory, and a group
// never spans the two halves (the host sends groups wider than half a row elsewhere).
template <typename T, typename TT, int VPT, int GV, int TPR>
__global__ void __launch_bounds__(reg_threads(reg_groups(VPT / TPR)), 1) rows_tma_wide_quant_kernel(const StreamArgs p) {
  constexpr bool GROUPED = GV != 0;
  constexpr int VW = VPT / TPR;                  // slots per warp
  constexpr int kRegGroups = reg_groups(VW);
  constexpr int kRegWarps = kRegRows * kRegGroups;
  constexpr int SR = kRegRows / TPR;             // rows per stage
  static_assert(TPR == 1 || TPR == 2, "one or two warps per row");
  extern __shared__ unsigned char smem_raw[];
  __shared__ float xch[kRegWarps][2];  // per warp: partial sum of squares, partial |y| maximum
  const Ring g = ring_setup(p, smem_raw, kRegRows, kRegWarps);
  const RowArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kRegWarps) {
    if (lane == 0)
      produce(p, g.smem, g.full, g.empty, g.wbar, g.w, g.resp, g.cbar, g.stage_row, SR, sizeof(T), sizeof(TT),
              kRegGroups);
    return;
  }
  const int grp = warp / kRegRows, wg = warp % kRegRows;  // consumer group, warp within the group
  const int wr = wg / TPR, hh = wg % TPR;                  // row within the stage, part of the row
  const int team = warp / TPR;
  constexpr int N = 256 * VPT;
  const int vb = hh * 32 * VW;           // first vector of this warp's part of the row
  const int hr = a.R >> 4;               // rotary vectors per half of the rotary block
  const bool rot = hh == TPR - 1 && lane >= 32 - 2 * hr;  // this lane's last-slot vector is a rotary one
  const bool is_lo = lane < 32 - hr;
  const int partner = is_lo ? lane + hr : lane - hr;
  const int pblk = is_lo ? lane - (32 - 2 * hr) : lane - (32 - hr);  // pairs 8 pblk .. 8 pblk + 7
  const int half = a.R >> 1;
  const uint4* ws = reinterpret_cast<const uint4*>(g.w) + vb;
  const int lg = GROUPED ? __ffs(a.group) - 1 : 0;  // log2 of the group size
  const int gv = GROUPED ? a.group >> 3 : 32 * VW;   // vectors per group
  const int G = GROUPED ? N >> lg : 1;
  const float fmax = a.fp8_max, rcp = __frcp_rn(a.fp8_max);
  const bool clamp = a.fp8_max != 448.0f;
  bool ok = mbar_wait(kWaitLimitNs, g.wbar, 0u);
  int slot = grp;  // stage k lives in slot k % S; this group takes stages grp, grp + 3, ...
  uint32_t phase = 0;
  for (;;) {
    ok = ok && mbar_wait(kWaitLimitNs, &g.full[slot], phase);
    if constexpr (TPR > 1) ok = team_all(ok, team, 32 * TPR);  // the partner looks at the stage only if both can
    if (!ok) {
      flag_failure(p.status);
      return;
    }
    const int32_t rs = g.stage_row[slot];
    if (rs < 0) break;  // end marker
    const int32_t r = rs + wr;
    const bool live = r < static_cast<int32_t>(a.rows);  // uniform over the row's warps
    const unsigned char* st = g.smem + static_cast<size_t>(slot) * p.stage_bytes;
    const uint4* xs = reinterpret_cast<const uint4*>(st + static_cast<size_t>(wr) * N * sizeof(T)) + vb;
    const int rel_slot = slot;
    slot += kRegGroups;
    if (slot >= p.stages) {
      slot -= p.stages;
      phase ^= 1u;
    }
    if (!live) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&g.empty[rel_slot]);
      continue;
    }
    uint4 xv[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k) xv[k] = xs[lane + 32 * k];
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VW; k += 2) {
      acc0 = sq_acc_mixed<T>(xv[k], acc0);
      acc1 = sq_acc_mixed<T>(xv[k + 1], acc1);
    }
    const float2 acc = add2(acc0, acc1);
    float ss = group_sum<32>(acc.x + acc.y);
    if constexpr (TPR > 1) {
      if (lane == 0) xch[warp][0] = ss;
      team_sync(team, 32 * TPR);
      ss = xch[team * TPR][0] + xch[team * TPR + 1][0];  // the same order in both warps
    }
    const float2 rstd2 = splat2(rstd_from_ss(ss, static_cast<float>(N), a.eps));
    // The last slot first: its rotary lanes read their partner's vector and their cos / sin entries
    // from the stage, which is released right after.
    // Per row: one running |y| maximum; per group: one per slot (fp32, before rounding: see norm8_max).
    float mk[GROUPED ? VW : 1];
#pragma unroll
    for (int k = 0; k < (GROUPED ? VW : 1); ++k) mk[k] = 0.f;
    {
      constexpr int k = VW - 1;
      float mrot = 0.f;  // the slot's maximum: its normalised values, or after rotation its rotated ones
      uint4 y = norm8_max<T>(xv[k], ws[lane + 32 * k], rstd2, mrot);
      if (rot) {
        mrot = 0.f;
        const uint4 yp = norm8<T>(xs[32 * k + partner], ws[32 * k + partner], rstd2);
        float2 c[4], sn[4];
        const int64_t off = static_cast<int64_t>(wr) * half + 8 * pblk;
        rows::load_table8<TT, true>(st + p.tab_off, off, c);
        rows::load_table8<TT, true>(st + p.tab_off + p.tab_block, off, sn);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 own = Elem<T>::unpack(rows::word(y, e)), other = Elem<T>::unpack(rows::word(yp, e));
          const float2 s2 = is_lo ? neg2(sn[e]) : sn[e];  // lo' = lo*c + hi*(-s), hi' = hi*c + lo*s
          const float2 v = add2(mul2(own, c[e]), mul2(other, s2));
          mrot = absmax4(mrot, v, make_float2(0.f, 0.f));
          rows::set_word(y, e, Elem<T>::pack(v));
        }
      }
      xv[k] = y;
      mk[GROUPED ? k : 0] = mrot;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[rel_slot]);  // everything this warp needs is in registers
    uint4* yrow = a.y != nullptr
                      ? reinterpret_cast<uint4*>(static_cast<T*>(a.y) + static_cast<int64_t>(r) * N) + vb
                      : nullptr;
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      if (k < VW - 1) xv[k] = norm8_max<T>(xv[k], ws[lane + 32 * k], rstd2, mk[GROUPED ? k : 0]);
      if (yrow != nullptr) st_stream16(yrow + lane + 32 * k, xv[k]);
    }
    uint2* qrow = reinterpret_cast<uint2*>(a.q + static_cast<int64_t>(r) * N) + vb;
    if constexpr (!GROUPED) {
      float m = warp_max(mk[0]);
      if constexpr (TPR > 1) {
        if (lane == 0) xch[warp][1] = m;
        team_sync(team, 32 * TPR);
        m = fmaxf(xch[team * TPR][1], xch[team * TPR + 1][1]);
      }
      const float sc = scale_of(fmaxf(round_to<T>(m), 1e-4f), fmax, rcp);
      const float rc = __frcp_rn(sc);
#pragma unroll
      for (int k = 0; k < VW; ++k) st_stream8(qrow + lane + 32 * k, codes8_rcp<T>(xv[k], rc, clamp, fmax));
      if (hh == 0 && lane == 0) a.scale[r] = sc;
    } else if constexpr (GV > 0) {
      // One group per (slot, segment of GV lanes). The slots are reduced in blocks of BLK (the
      // largest power of two dividing VW); after a block's reduce-scatter every lane owns NF of its
      // groups: it computes their scales and reciprocals once and writes the scales; each lane then
      // fetches its slots' scale and reciprocal from the owner.
      static_assert(GV <= 32 && (GV & (GV - 1)) == 0, "reduce-scatter shape");
      constexpr int BLK = VW & -VW, NB = VW / BLK;
      constexpr int NF = BLK >= GV ? BLK / GV : 1;
      const int j = lane & (GV - 1), sgm = lane / GV;
      float* srow = a.scale + static_cast<int64_t>(r) * (N / (8 * GV)) + hh * (VW * 32 / GV);
      float sgv[NB][NF], rgv[NB][NF];
#pragma unroll
      for (int bk = 0; bk < NB; ++bk) {
        float m[BLK];
#pragma unroll
        for (int i = 0; i < BLK; ++i) m[i] = mk[bk * BLK + i];
        if constexpr (GV > 1) seg_reduce_scatter<BLK, GV / 2, BLK>(m, lane);
#pragma unroll
        for (int i = 0; i < NF; ++i) {
          sgv[bk][i] = scale_of(fmaxf(round_to<T>(m[i]), 1e-4f), fmax, rcp);
          rgv[bk][i] = __frcp_rn(sgv[bk][i]);
          const int k = bk * BLK + (BLK >= GV ? i + NF * j : (j * BLK) / GV);
          if (BLK >= GV || (j & (GV / BLK - 1)) == 0) srow[k * (32 / GV) + sgm] = sgv[bk][i];
        }
      }
#pragma unroll
      for (int k = 0; k < VW; ++k) {
        const int bk = k / BLK, kb = k % BLK;
        const int src = sgm * GV + (BLK >= GV ? kb / NF : kb * (GV / BLK));
        const float rg = __shfl_sync(0xffffffffu, rgv[bk][kb % NF], src);
        st_stream8(qrow + lane + 32 * k, codes8_rcp<T>(xv[k], rg, clamp, fmax));
      }
    } else {
      // Group maxima: within a slot a group is gv consecutive lanes (gv <= 32) ...
#pragma unroll
      for (int k = 0; k < VW; ++k)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
          if (o < gv) mk[k] = fmaxf(mk[k], __shfl_xor_sync(0xffffffffu, mk[k], o));
      // ... and a group of more than 32 vectors spans gv / 32 consecutive slots.
#pragma unroll
      for (int d = 1; d < VW; d <<= 1)
        if (32 * d < gv) {
#pragma unroll
          for (int k = 0; k < VW; ++k)
            if ((k & d) == 0 && (k | d) < VW) mk[k] = mk[k | d] = fmaxf(mk[k], mk[k | d]);
        }
      float* srow = a.scale + static_cast<int64_t>(r) * G;
#pragma unroll
      for (int k = 0; k < VW; ++k) {
        const float sg = scale_of(fmaxf(round_to<T>(mk[k]), 1e-4f), fmax, rcp);
        const float rg = __frcp_rn(sg);
        st_stream8(qrow + lane + 32 * k, codes8_rcp<T>(xv[k], rg, clamp, fmax));
        const int col = 8 * (vb + lane + 32 * k);
        if ((col & (a.group - 1)) == 0) srow[col >> lg] = sg;  // the group's first vector
      }
    }
  }
}

// ------------------------------------------------------------------ wide rows, RMSNorm, registers
// RMSNorm forward for rows of 1024 <= N <= 4096 with the consumer layout of the LayerNorm kernel
// below (consumer groups taking stages in turn, one CTA per SM, two warps per row above 2048
// columns): the warp copies its part of the row into registers and releases the stage, adds its
// squares in four chains, and writes y = dtype((x * rstd) * w) from the registers.
template <typename T, int VPT, int TPR>
__global__ void __launch_bounds__(reg_threads(reg_groups(VPT / TPR)), 1) rows_tma_reg_fwd_kernel(const StreamArgs p) {
  constexpr int VW = VPT / TPR;
  constexpr int kRegGroups = reg_groups(VW);
  constexpr int kRegWarps = kRegRows * kRegGroups;
  constexpr int SR = kRegRows / TPR;
  static_assert(TPR == 1 || TPR == 2, "one or two warps per row");
  extern __shared__ unsigned char smem_raw[];
  __shared__ float xch[kRegWarps];  // per warp: partial sum of squares
  const Ring g = ring_setup(p, smem_raw, kRegRows, kRegWarps);
  const RowArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kRegWarps) {
    if (lane == 0)
      produce(p, g.smem, g.full, g.empty, g.wbar, g.w, g.resp, g.cbar, g.stage_row, SR, sizeof(T), 2, kRegGroups);
    return;
  }
  const int grp = warp / kRegRows, wg = warp % kRegRows;
  const int wr = wg / TPR, hh = wg % TPR;
  const int team = warp / TPR;
  const int N = a.N, nv = N >> 3;
  const int vb = hh * 32 * VW;  // first vector of this warp's part of the row
  const float fN = static_cast<float>(N);
  const uint4* ws = reinterpret_cast<const uint4*>(g.w) + vb;
  bool ok = mbar_wait(kWaitLimitNs, g.wbar, 0u);
  int slot = grp;
  uint32_t phase = 0;
  for (;;) {
    ok = ok && mbar_wait(kWaitLimitNs, &g.full[slot], phase);
    if constexpr (TPR > 1) ok = team_all(ok, team, 32 * TPR);
    if (!ok) {
      flag_failure(p.status);
      return;
    }
    const int32_t rs = g.stage_row[slot];
    if (rs < 0) break;  // end marker
    const int32_t r = rs + wr;
    const bool live = r < static_cast<int32_t>(a.rows);  // uniform over the row's warps
    const uint4* xs = reinterpret_cast<const uint4*>(g.smem + static_cast<size_t>(slot) * p.stage_bytes +
                                                     static_cast<size_t>(wr) * N * sizeof(T)) + vb;
    uint4 xv[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k)
      xv[k] = (live && vb + lane + 32 * k < nv) ? xs[lane + 32 * k] : make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[slot]);  // the row is in registers: release the stage
    slot += kRegGroups;
    if (slot >= p.stages) {
      slot -= p.stages;
      phase ^= 1u;
    }
    if (!live) continue;
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int k = 0; k < VW; ++k) acc[k & 3] = sq_acc_mixed<T>(xv[k], acc[k & 3]);
    const float2 sum = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
    float ss = group_sum<32>(sum.x + sum.y);
    if constexpr (TPR > 1) {
      if (lane == 0) xch[warp] = ss;
      team_sync(team, 32 * TPR);
      ss = xch[team * TPR] + xch[team * TPR + 1];  // the same order in both warps
    }
    const float rstd = rstd_from_ss(ss, fN, a.eps);
    if (a.rstd != nullptr && hh == 0 && lane == 0) a.rstd[r] = rstd;
    const float2 rstd2 = splat2(rstd);
    uint4* yrow = reinterpret_cast<uint4*>(static_cast<T*>(a.y) + static_cast<int64_t>(r) * N) + vb;
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const int v = lane + 32 * k;
      if (vb + v < nv) st_stream16(yrow + v, norm8<T>(xv[k], ws[v], rstd2));
    }
  }
}

// ------------------------------------------------------------------ wide rows, LayerNorm
// LayerNorm forward ("ledger.py" (Ch.13 ledger), layer_norm) for rows of 1024 <= N <= 4096, with the
// consumer layout of the FP8 kernel above: consumer groups of four warps take the stages in turn (one
// CTA per SM), TPR warps per row (two for rows longer than 2048, each holding one contiguous half),
// the gain and bias rows staged once per CTA. A warp copies its part of the row into registers
// (VPT / TPR 16-byte vectors per lane) and releases the stage at once; then three passes over the
// registers: the mean, the variance of the deviations (no E[x^2] - E[x]^2 cancellation), and
// y = dtype(((x - mean) * rstd) * g + b) with each step rounded as the definition's fp32 ops. With
// two warps per row their partial sums meet in shared memory, added in the same order by both.
template <typename T, int VPT, int TPR>
__global__ void __launch_bounds__(reg_threads(reg_groups(VPT / TPR)), 1) rows_tma_ln_kernel(const StreamArgs p) {
  constexpr int VW = VPT / TPR;
  constexpr int kRegGroups = reg_groups(VW);
  constexpr int kRegWarps = kRegRows * kRegGroups;
  constexpr int SR = kRegRows / TPR;
  static_assert(TPR == 1 || TPR == 2, "one or two warps per row");
  extern __shared__ unsigned char smem_raw[];
  __shared__ float xch[kRegWarps][2];  // per warp: partial sum, partial sum of squared deviations
  const Ring g = ring_setup(p, smem_raw, kRegRows, kRegWarps);
  const RowArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kRegWarps) {
    if (lane == 0)
      produce(p, g.smem, g.full, g.empty, g.wbar, g.w, g.resp, g.cbar, g.stage_row, SR, sizeof(T), 2, kRegGroups);
    return;
  }
  const int grp = warp / kRegRows, wg = warp % kRegRows;
  const int wr = wg / TPR, hh = wg % TPR;
  const int team = warp / TPR;
  const int N = a.N, nv = N >> 3;
  const int vb = hh * 32 * VW;  // first vector of this warp's part of the row
  const float fN = static_cast<float>(N);
  const uint4* gs = reinterpret_cast<const uint4*>(g.w) + vb;
  const uint4* bs = p.b_bytes > 0 ? reinterpret_cast<const uint4*>(g.w + p.w_bytes) + vb : nullptr;
  bool ok = mbar_wait(kWaitLimitNs, g.wbar, 0u);
  int slot = grp;
  uint32_t phase = 0;
  for (;;) {
    ok = ok && mbar_wait(kWaitLimitNs, &g.full[slot], phase);
    if constexpr (TPR > 1) ok = team_all(ok, team, 32 * TPR);
    if (!ok) {
      flag_failure(p.status);
      return;
    }
    const int32_t rs = g.stage_row[slot];
    if (rs < 0) break;  // end marker
    const int32_t r = rs + wr;
    const bool live = r < static_cast<int32_t>(a.rows);  // uniform over the row's warps
    const uint4* xs = reinterpret_cast<const uint4*>(g.smem + static_cast<size_t>(slot) * p.stage_bytes +
                                                     static_cast<size_t>(wr) * N * sizeof(T)) + vb;
    uint4 xv[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k)
      xv[k] = (live && vb + lane + 32 * k < nv) ? xs[lane + 32 * k] : make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[slot]);  // the row is in registers: release the stage
    slot += kRegGroups;
    if (slot >= p.stages) {
      slot -= p.stages;
      phase ^= 1u;
    }
    if (!live) continue;
    // Sums with four independent chains (the absent vectors are zeros and add nothing).
    float2 s0 = make_float2(0.f, 0.f), s1 = s0, s2 = s0, s3 = s0;
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      float2& sa = (k & 1) ? s1 : s0;
      float2& sb = (k & 1) ? s3 : s2;
      sa = Mixed<T>::add(xv[k].y, Mixed<T>::add(xv[k].x, sa));
      sb = Mixed<T>::add(xv[k].w, Mixed<T>::add(xv[k].z, sb));
    }
    const float2 st = add2(add2(s0, s1), add2(s2, s3));
    float sum = group_sum<32>(st.x + st.y);
    if constexpr (TPR > 1) {
      if (lane == 0) xch[warp][0] = sum;
      team_sync(team, 32 * TPR);
      sum = xch[team * TPR][0] + xch[team * TPR + 1][0];
    }
    const float mean = div_n(sum, fN);
    const float2 nmean2 = splat2(-mean);  // x - mean as x * 1 + (-mean): one rounding, as the subtraction
    float2 q0 = make_float2(0.f, 0.f), q1 = q0, q2 = q0, q3 = q0;
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      if (vb + lane + 32 * k >= nv) continue;
      const float2 c0 = Mixed<T>::add(xv[k].x, nmean2), c1 = Mixed<T>::add(xv[k].y, nmean2);
      const float2 c2 = Mixed<T>::add(xv[k].z, nmean2), c3 = Mixed<T>::add(xv[k].w, nmean2);
      float2& qa = (k & 1) ? q1 : q0;
      float2& qb = (k & 1) ? q3 : q2;
      qa = fma2(c0, c0, fma2(c1, c1, qa));
      qb = fma2(c2, c2, fma2(c3, c3, qb));
    }
    const float2 qt = add2(add2(q0, q1), add2(q2, q3));
    float qs = group_sum<32>(qt.x + qt.y);
    if constexpr (TPR > 1) {
      if (lane == 0) xch[warp][1] = qs;
      team_sync(team, 32 * TPR);
      qs = xch[team * TPR][1] + xch[team * TPR + 1][1];
    }
    const float var = div_n(qs, fN);
    const float2 rstd2 = splat2(__frcp_rn(__fsqrt_rn(__fadd_rn(var, a.eps))));
    uint4* yrow = reinterpret_cast<uint4*>(static_cast<T*>(a.y) + static_cast<int64_t>(r) * N) + vb;
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const int v = lane + 32 * k;
      if (vb + v >= nv) continue;
      const uint4 gv = gs[v];
      const uint4 bv = bs != nullptr ? bs[v] : make_uint4(0u, 0u, 0u, 0u);
      uint4 out;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 c = Mixed<T>::add(rows::word(xv[k], e), nmean2);
        const float2 n = mul2(mul2(c, rstd2), Elem<T>::unpack(rows::word(gv, e)));
        rows::set_word(out, e, Elem<T>::pack(Mixed<T>::add(rows::word(bv, e), n)));  // n + bias, one rounding
      }
      st_stream16(yrow + v, out);
    }
  }
}

// ---------------------------------------------------------------------------------- host side
// `budget`: shared-memory bytes for the ring (0: two CTAs per SM when stages are small, else one);
// `inflight`: bytes the producer keeps in flight; `groups`: consumer groups that take the stages in
// turn (stage k goes to group k % groups).
//
// With several groups the ring holds a multiple of `groups` stages, so that a slot always belongs to
// the same group. A consumer waits for stage k on its slot's full barrier by phase parity, which
// cannot tell the phase of stage k from that of stage k - 2S: the wait is only sound if the slot's
// previous use, stage k - S, has completed. The group consumed stage k - S itself, in order, before
// it waits for stage k, so it has.
template <typename K>
bool launch_stream(K kern, int threads, StreamArgs p, int stage_rows, int x_row_bytes, int tab_row_bytes,
                   cudaStream_t s, int extra_bytes = 0, int budget = 0, int inflight = 48 * 1024, int groups = 1) {
  const RowArgs& a = p.a;
  p.status = device_status_ptr();
  p.tab_block = ((stage_rows * tab_row_bytes) + 127) & ~127;
  p.tab_off = (stage_rows * x_row_bytes + 127) & ~127;
  p.stage_bytes = p.tab_off + 2 * p.tab_block;
  // Two CTAs per SM when stages are small (a four-row stage of 4096-wide rows with its table rows
  // still fits three times); as many stages as fit, at most 8.
  if (budget == 0) budget = p.stage_bytes <= 36 * 1024 ? 110 * 1024 : 220 * 1024;
  p.stages = (budget - static_cast<int>(ring_bytes(0, 0, p.w_bytes)) - extra_bytes - 8) / (p.stage_bytes + 20);
  const int cap = groups > 1 ? 12 : 8;
  if (p.stages > cap) p.stages = cap;
  p.stages -= p.stages % groups;
  if (p.stages < 2 || p.stages < groups) return false;
  // Keep about `inflight` bytes in flight per CTA (at least two stages), never more than the ring.
  p.depth = (inflight + p.stage_bytes - 1) / p.stage_bytes;
  if (p.depth < 2) p.depth = 2;
  if (p.depth > p.stages) p.depth = p.stages;
  const size_t smem = ring_bytes(p.stages, p.stage_bytes, p.w_bytes) + extra_bytes;
  if (smem > 227 * 1024) return false;
  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem)) return false;
  // One CTA per stage of rows. Only the CTAs that fit on the GPU at once start; they take over the
  // rest of the grid stage by stage (cluster launch control), so the grid is not a wave count.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>((a.rows + stage_rows - 1) / stage_rows));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess;
}

template <typename T, typename TT, int MODE, int LPR, int HS, int TS, int G = 1>
bool launch_narrow(const RowArgs& a, cudaStream_t s) {
  StreamArgs p{};
  p.a = a;
  constexpr int SR = (kConsumerWarps / G) * (32 / LPR);
  return launch_stream(rows_tma_kernel<T, TT, MODE, LPR, HS, TS, G>, kThreads, p, SR,
                       a.N * static_cast<int>(sizeof(T)), (a.R / 2) * static_cast<int>(sizeof(TT)), s, 0, 0,
                       48 * 1024, G);
}

template <typename T, typename TT, int MODE>
bool dispatch_narrow(const RowArgs& a, cudaStream_t s) {
  const int hv = (a.N - a.R) / 8, th = a.R / 16;
#define FQ_TMA_TRY(L, H, S)                                       \
  if (hv <= (L) * (H) && th <= (L) * (S) && ((S) > 0 || th == 0)) \
    return launch_narrow<T, TT, MODE, L, H, S>(a, s);
  if constexpr (MODE == MODE_FWD) {
    FQ_TMA_TRY(8, 2, 0) FQ_TMA_TRY(16, 2, 0) FQ_TMA_TRY(32, 2, 0)
  } else {
    FQ_TMA_TRY(8, 0, 1)
    // fp16 rows of up to 128 head and 64 rotary columns (the 65536 x 192 workload: 16 head and 4 rotary
    // vectors): four lanes per row fill every slot and need two shuffle levels, 10.85 against 11.11 us
    // for eight lanes; consumer groups that take the stages in turn make the work units finer for
    // the 304 resident CTAs: four groups (16-row stages, 4096 units) 10.28 us, two (32-row stages)
    // 10.43-10.45, one (64-row stages, 1024 units) 11.00. (bf16 would spill at two CTAs per SM in this
    // shape.)
    if constexpr (std::is_same<T, __half>::value) {
      if (hv <= 16 && th <= 4) return launch_narrow<T, TT, MODE, 4, 4, 1, 4>(a, s);
    }
    FQ_TMA_TRY(8, 2, 1) FQ_TMA_TRY(16, 2, 1) FQ_TMA_TRY(32, 2, 1) FQ_TMA_TRY(32, 4, 1)
  }
#undef FQ_TMA_TRY
  return false;
}

}  // namespace

bool launch_layernorm_tma(const RowArgs& a, int dtype, cudaStream_t s) {
  if (a.rows < 4096 || a.rows > 0x7fffffffLL - 256) return false;
  if (a.token_stride != a.N || a.H != 1 || a.N < 1024 || a.N > 4096) return false;
  StreamArgs p{};
  p.a = a;
  p.a.R = 0;
  const int xrow = a.N * 2;
  p.w_bytes = xrow;                           // the gain row
  p.b_bytes = a.bias != nullptr ? xrow : 0;   // the bias row, right after it
#define FQ_LN_K(T, V, TPR)                                                                                 \
  launch_stream(rows_tma_ln_kernel<T, V, TPR>, reg_threads(reg_groups((V) / (TPR))), p, kRegRows / (TPR), xrow, \
                0, s, p.b_bytes, 220 * 1024, 96 * 1024, reg_groups((V) / (TPR)))
#define FQ_LN(V)                                                                                      \
  return dtype == DT_BF16 ? FQ_LN_K(__nv_bfloat16, V, (V) == 16 ? 2 : 1) : FQ_LN_K(__half, V, (V) == 16 ? 2 : 1)
  const int nv = a.N / 8;
  if (nv <= 4 * 32) FQ_LN(4);
  if (nv <= 8 * 32) FQ_LN(8);
  FQ_LN(16);
#undef FQ_LN
#undef FQ_LN_K
}

bool launch_rows_tma(const RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s) {
  // Small problems are launch-bound: the generic kernel. Row indices and row + stage stay in int32.
  if (a.rows < 4096 || a.rows > 0x7fffffffLL - 256) return false;
  if (a.token_stride != a.N || a.H != 1) return false;       // contiguous rows only
  if (mode != MODE_FWD && mode != MODE_ROPE && mode != MODE_ROPE_QUANT) return false;
  if (mode != MODE_FWD && a.R > 0 && table_dtype != DT_FP32 && table_dtype != dtype) return false;
  if (mode != MODE_FWD && a.N >= 1024) {
    StreamArgs p{};
    p.a = a;
    const int xrow = a.N * 2;
    p.w_bytes = xrow;
    const int tsz = (a.R > 0 && table_dtype == DT_FP32) ? 4 : 2;
    const int trow = (a.R / 2) * tsz;
    const int extra = (mode == MODE_ROPE_QUANT && a.group > 0) ? kWideWarps * 3 * (a.N / a.group) * 4 : 0;
    const bool quant = mode == MODE_ROPE_QUANT;
    // Quantising rows of 1024, 2048, 3072 or 4096 with rope_dim <= 256 and a power-of-two group
    // size (or one scale per row): the register-resident kernel, one CTA per SM.
    const int vpt = a.N / 256;
    const bool pow2_group = a.group == 0 || (a.group >= 8 && (a.group & (a.group - 1)) == 0 && a.N % a.group == 0);
    const bool grouped = a.group > 0 && a.group < a.N;  // a group of the whole row is the per-row scale
    // FQ_ROWS_KERNEL=staged keeps these on the shared-memory kernel below (diagnostic switch: both
    // compute the same result).
    const char* sel = getenv("FQ_ROWS_KERNEL");
    const bool staged = sel != nullptr && std::string(sel) == "staged";
    if (quant && !staged && a.N % 256 == 0 && (vpt == 4 || vpt == 8 || vpt == 12 || vpt == 16) && a.R <= 256 &&
        a.R % 16 == 0 && pow2_group) {
// Bytes in flight per CTA for the FP8 kernel: the whole ring (ten two-row stages of 4096-wide rows).
// Measured on 4096 x 4096: 96 KB (six stages) 10.58 us, 136 KB 10.48, the whole ring 10.45; the
// RMSNorm forward and LayerNorm kernels are faster at 96 KB (21.19 against 21.34 us, 11.56 against
// 11.87).
constexpr int kQuantInflight = 176 * 1024;
#define FQ_REG_K2(T, TT, V, GV, TPR)                                                                         \
  return launch_stream(rows_tma_wide_quant_kernel<T, TT, V, GV, TPR>, reg_threads(reg_groups((V) / (TPR))), p, \
                       kRegRows / (TPR), xrow, trow, s, 0, 220 * 1024, kQuantInflight, reg_groups((V) / (TPR)));
// Rows of 4096: two warps per row, so that three or four consumer groups fit the registers. (A power-of-two
// group narrower than the row is at most half of it, so no group spans the two warps; a group of the
// whole row takes the per-row kernel, which does not read the group size.)
#define FQ_REG_K(T, TT, V, GV)                                                      \
  {                                                                                 \
    if constexpr ((V) == 16) {                                                      \
      FQ_REG_K2(T, TT, V, GV, 2)                                                    \
    } else {                                                                        \
      FQ_REG_K2(T, TT, V, GV, 1)                                                    \
    }                                                                               \
  }
#define FQ_REG(T, TT, V)                                         \
  if (vpt == (V)) {                                              \
    if (!grouped) FQ_REG_K(T, TT, V, 0)                          \
    if (a.group == 128) FQ_REG_K(T, TT, V, 16)                   \
    FQ_REG_K(T, TT, V, -1)                                       \
  }
#define FQ_REG_T(T, TT) FQ_REG(T, TT, 4) FQ_REG(T, TT, 8) FQ_REG(T, TT, 12) FQ_REG(T, TT, 16)
      if (dtype == DT_BF16) {
        if (tsz == 4) {
          FQ_REG_T(__nv_bfloat16, float)
        } else {
          FQ_REG_T(__nv_bfloat16, __nv_bfloat16)
        }
      } else if (tsz == 4) {
        FQ_REG_T(__half, float)
      } else {
        FQ_REG_T(__half, __half)
      }
#undef FQ_REG_T
#undef FQ_REG
#undef FQ_REG_K
#undef FQ_REG_K2
    }
#define FQ_WIDE(T, TT)                                                                                      \
  return quant ? launch_stream(rows_tma_wide_rope_kernel<T, TT, true>, kWideThreads, p, kWideWarps, xrow, trow, s, \
                               extra)                                                                       \
               : launch_stream(rows_tma_wide_rope_kernel<T, TT, false>, kWideThreads, p, kWideWarps, xrow, trow, s)
    if (dtype == DT_BF16) {
      if (tsz == 4) FQ_WIDE(__nv_bfloat16, float);
      FQ_WIDE(__nv_bfloat16, __nv_bfloat16);
    }
    if (tsz == 4) FQ_WIDE(__half, float);
    FQ_WIDE(__half, __half);
#undef FQ_WIDE
  }
  if (mode == MODE_ROPE_QUANT) return false;  // narrower quantising rows: the generic kernel
  if (mode == MODE_FWD && a.N >= 1024) {
    StreamArgs p{};
    p.a = a;
    p.a.R = 0;
    const int xrow = a.N * 2;
    p.w_bytes = xrow;  // N % 8 == 0 and a 16-byte aligned w: a legal bulk copy
    const char* sel = getenv("FQ_ROWS_KERNEL");
    if (a.N <= 4096 && !(sel != nullptr && std::string(sel) == "staged")) {
#define FQ_RF_K(T, V, TPR)                                                                                 \
  launch_stream(rows_tma_reg_fwd_kernel<T, V, TPR>, reg_threads(reg_groups((V) / (TPR))), p, kRegRows / (TPR), \
                xrow, 0, s, 0, 220 * 1024, 96 * 1024, reg_groups((V) / (TPR)))
#define FQ_RF(V)                                                                                                  \
  return dtype == DT_BF16 ? FQ_RF_K(__nv_bfloat16, V, (V) == 16 ? 2 : 1) : FQ_RF_K(__half, V, (V) == 16 ? 2 : 1)
      const int nv = a.N / 8;
      if (nv <= 4 * 32) FQ_RF(4);
      if (nv <= 8 * 32) FQ_RF(8);
      FQ_RF(16);
#undef FQ_RF
#undef FQ_RF_K
    }
    if (dtype == DT_BF16)
      return launch_stream(rows_tma_wide_fwd_kernel<__nv_bfloat16>, kWideThreads, p, kWideWarps, xrow, 0, s);
    return launch_stream(rows_tma_wide_fwd_kernel<__half>, kWideThreads, p, kWideWarps, xrow, 0, s);
  }
  if (mode == MODE_FWD) {
    if (dtype == DT_BF16) return dispatch_narrow<__nv_bfloat16, __nv_bfloat16, MODE_FWD>(a, s);
    return dispatch_narrow<__half, __half, MODE_FWD>(a, s);
  }
  if (a.R == 0) {
    if (dtype == DT_BF16) return dispatch_narrow<__nv_bfloat16, __nv_bfloat16, MODE_ROPE>(a, s);
    return dispatch_narrow<__half, __half, MODE_ROPE>(a, s);
  }
  if (dtype == DT_BF16) {
    if (table_dtype == DT_FP32) return dispatch_narrow<__nv_bfloat16, float, MODE_ROPE>(a, s);
    return dispatch_narrow<__nv_bfloat16, __nv_bfloat16, MODE_ROPE>(a, s);
  }
  if (table_dtype == DT_FP32) return dispatch_narrow<__half, float, MODE_ROPE>(a, s);
  return dispatch_narrow<__half, __half, MODE_ROPE>(a, s);
}

}  // namespace fq
