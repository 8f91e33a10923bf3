// fq_prologue.cu -- the QK-Norm + RoPE + FP8 attention prologue ("case_norm_rope_quant.py" (Ch.28),
// module docstring) for head_dim 128 with the whole head rotated, as a TMA-fed persistent kernel.
//
// Data movement. The rows are cut into chunks of SR consecutive (token, head) rows, one per CTA of
// the grid. The CTAs that are resident take over the chunks of CTAs that have not started yet
// through cluster launch control (a hardware work queue: no counter in global memory), so every
// SM keeps streaming until the last chunk is taken and the CTAs finish together. One producer
// lane streams its chunks through a ring of shared-memory stages, one chunk per stage: two 2-D
// tensor TMA loads (cp.async.bulk.tensor, 128-byte swizzle) bring the first and second halves of
// the SR rows (the NeoX "lo" and "hi" halves) and two 1-D bulk copies bring the cos and sin rows
// of the tokens those rows belong to; an mbarrier counts the bytes. Bytes in flight do not depend
// on registers or occupancy. x is read from HBM once; each table row once per stage that needs it
// (L2 serves repeats); the two norm weights once per CTA (shared memory, fp32, in a lane-permuted
// layout). Codes and scales go straight to global memory with evict-first stores.
//
// Work layout. Eight consumer warps, four lanes per row (eight rows per warp, one row per lane group
// per stage). Lane j of a row holds the NeoX pairs 16j..16j+15 of both halves, so every pair
// (p, p+64) sits in one thread: no shuffle and no shared-memory round trip for the rotation. The
// swizzle makes the four lanes' 16-byte reads of two neighbouring rows hit disjoint banks. Each
// lane stores its 16 contiguous codes of each half with one 16-byte store.
//
// Arithmetic (the oracle's cast points, with two hardware shortcuts that stay far inside the
// parity tolerances -- scale within 1e-5 relative, codes at most one step apart on at most 0.1%):
//   ss = sum x^2 (fp32) -> rstd = rsqrt(ss/128 + eps) with the hardware rsqrt approximation (at
//   most 2 ulp, as torch's own CUDA rsqrt; ss/128 is exact as ss * 2^-7); n = (x*rstd)*w;
//   lo' = lo*c - hi*s, hi' = hi*c + lo*s (the compiler may fuse a product into the sum);
//   scale = RN(max(amax, 1e-4)/fp8_max) (correctly rounded); q = e4m3(RN(y * RN(1/scale))).
// A perturbation of one or two fp32 ulps moves a code only when y/scale sits at an e4m3 rounding
// boundary, so the codes match the oracle's true division except on a vanishing fraction.
//
// Waits are bounded: a wait that has not completed after ~1 s of %globaltimer time sets bit 0 of
// the device status word and the kernel stops issuing and consuming work (waiting, again bounded,
// for the copies it has in flight) instead of trapping.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "fq_device.cuh"
#include "fq_internal.h"
#include "fq_sync.cuh"

namespace fq {
namespace {

constexpr int kD = 128;                                  // head_dim handled here
constexpr int kLPR = 4;                                  // lanes per row
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;      // + one producer warp
constexpr int kGroupsPerHalf = (kConsumerWarps / 2) * (32 / kLPR);  // lane groups in one consumer half
// Rows per stage (SR) is a template parameter: 64 for long row ranges per CTA, 32 when a CTA has
// only a few stages to do (shorter pipeline fill and drain). Each lane group takes SR / 32 rows of
// every stage its half consumes. One half of a stage's x (the NeoX lo or hi half) is SR * 128 bytes.
template <int SR>
__host__ __device__ constexpr int half_tile() { return SR * (kD / 2) * 2; }

struct PrologueArgs {
  const void* wq;
  const void* wk;
  const void* cos;
  const void* sin;
  uint8_t* q;
  float* scale;
  unsigned int* status;
  uint64_t magic;        // t = (r * magic) >> shift == r / H for r < 2^31
  int32_t shift;
  int32_t rows;          // T * H
  int32_t H, Hq;
  float inv_h;           // RN(1/H), for floor(x / H) with x < 2^21
  float eps, fp8_max, rcp_fp8_max;
  int32_t stages;        // ring depth
  int32_t stage_bytes;   // 2 half tiles + 2 table blocks, multiple of 1024
  int32_t tab_block;     // bytes of one table block (cos or sin)
  int32_t depth;         // the producer keeps at most this many stages in flight
};

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds16f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// Table entries 8m..8m+7 of the lane's 16 (pairs 16j+8m..16j+8m+7 of one table row) -> 4 float2.
template <typename TT>
__device__ __forceinline__ void lds_table8(uint32_t addr, int m, float2 (&v)[4]) {
  if constexpr (sizeof(TT) == 4) {
    const float4 f0 = lds16f(addr + 32 * m), f1 = lds16f(addr + 32 * m + 16);
    v[0] = make_float2(f0.x, f0.y);
    v[1] = make_float2(f0.z, f0.w);
    v[2] = make_float2(f1.x, f1.y);
    v[3] = make_float2(f1.z, f1.w);
  } else {
    const uint4 u = lds16(addr + 16 * m);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = Elem<TT>::unpack(word(u, e));
  }
}

// One (token, head) row of a stage, by the four lanes of a lane group: shared-memory x, table and
// weight entries in, e4m3 codes and the fp32 scale out. `l` is the row within the stage.
template <typename T, typename TT, int SR>
__device__ __forceinline__ void prologue_row(const PrologueArgs& a, uint32_t st, int l, int j, int rev,
                                             uint32_t wbase, int32_t rs, int32_t r1, int32_t tf, bool clamp) {
  constexpr int kTabRow = (kD / 2) * static_cast<int>(sizeof(TT));
  const int sw = l & 7;  // 128-byte swizzle phase of this row
  const bool live = l < r1 - rs;
  const int32_t xh = (rs - tf * a.H) + l;                                             // head index from token tf
  const int32_t dt = static_cast<int32_t>((static_cast<float>(xh) + 0.5f) * a.inv_h);  // floor(xh / H)
  const int32_t h = xh - dt * a.H;
  const int32_t r = rs + l;
  const uint32_t xrow = st + l * 128;
  const uint4 xl0 = lds16(xrow + (((2 * j + rev) ^ sw) << 4));
  const uint4 xl1 = lds16(xrow + (((2 * j + (rev ^ 1)) ^ sw) << 4));
  const uint4 xh0 = lds16(xrow + half_tile<SR>() + (((2 * j + rev) ^ sw) << 4));
  const uint4 xh1 = lds16(xrow + half_tile<SR>() + (((2 * j + (rev ^ 1)) ^ sw) << 4));
  const uint32_t tcos = st + 2 * half_tile<SR>() + dt * kTabRow + j * (16 * static_cast<int>(sizeof(TT)));
  const uint32_t wa = wbase + (h >= a.Hq ? 512u : 0u);  // the k weights follow the q weights

  float2 lo[8], hi[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lo[e] = Elem<T>::unpack(word(xl0, e));
    lo[4 + e] = Elem<T>::unpack(word(xl1, e));
    hi[e] = Elem<T>::unpack(word(xh0, e));
    hi[4 + e] = Elem<T>::unpack(word(xh1, e));
  }
  // Sum of squares with four independent accumulators (short dependency chains).
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    acc[0] = fma2(lo[i], lo[i], acc[0]);
    acc[1] = fma2(lo[i + 1], lo[i + 1], acc[1]);
    acc[2] = fma2(hi[i], hi[i], acc[2]);
    acc[3] = fma2(hi[i + 1], hi[i + 1], acc[3]);
  }
  const float2 acc2 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
  const float ss = group_sum<kLPR>(acc2.x + acc2.y);
  // ss/128 is exact as a multiplication by 2^-7; rsqrt is the hardware approximation.
  const float rstd = rsqrtf(__fadd_rn(__fmul_rn(ss, 0.0078125f), a.eps));
  const float2 rstd2 = splat2(rstd);
  float pm[4];  // partial |y| maxima (four independent chains)
  // Normalise and rotate eight pairs at a time (weights and table entries loaded per sub-chunk).
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int sm = m ^ rev;  // the sub-chunk this step works on
    float2 wl[4], wh[4], c[4], s[4];
#pragma unroll
    for (int q4 = 0; q4 < 2; ++q4) {
      const float4 fl = lds16f(wa + (2 * sm + q4) * 64);
      const float4 fh = lds16f(wa + 256 + (2 * sm + q4) * 64);
      wl[2 * q4] = make_float2(fl.x, fl.y);
      wl[2 * q4 + 1] = make_float2(fl.z, fl.w);
      wh[2 * q4] = make_float2(fh.x, fh.y);
      wh[2 * q4 + 1] = make_float2(fh.z, fh.w);
    }
    lds_table8<TT>(tcos, sm, c);
    lds_table8<TT>(tcos + a.tab_block, sm, s);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 4 * m + e;
      const float2 nl = mul2(mul2(lo[i], rstd2), wl[e]);
      const float2 nh = mul2(mul2(hi[i], rstd2), wh[e]);
      lo[i] = sub2(mul2(nl, c[e]), mul2(nh, s[e]));
      hi[i] = add2(mul2(nh, c[e]), mul2(nl, s[e]));
    }
    pm[2 * m] = absmax4(absmax4(0.f, lo[4 * m], hi[4 * m]), lo[4 * m + 1], hi[4 * m + 1]);
    pm[2 * m + 1] = absmax4(absmax4(0.f, lo[4 * m + 2], hi[4 * m + 2]), lo[4 * m + 3], hi[4 * m + 3]);
  }
  float amax;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(amax) : "f"(pm[0]), "f"(pm[1]), "f"(pm[2]));
  amax = fmaxf(amax, pm[3]);
  amax = fmaxf(group_max<kLPR>(amax), 1e-4f);
  // scale = RN(amax / fp8_max) via the correctly rounded reciprocal and one correction.
  const float s0 = __fmul_rn(amax, a.rcp_fp8_max);
  const float sc = __fmaf_rn(__fmaf_rn(-s0, a.fp8_max, amax), a.rcp_fp8_max, s0);
  const float rc = __frcp_rn(sc);
  uint32_t ql[4], qh[4];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    float2 a0 = mul2(lo[i], splat2(rc)), a1 = mul2(lo[i + 1], splat2(rc));
    float2 b0 = mul2(hi[i], splat2(rc)), b1 = mul2(hi[i + 1], splat2(rc));
    if (clamp) {
      a0 = make_float2(clamp_abs(a0.x, a.fp8_max), clamp_abs(a0.y, a.fp8_max));
      a1 = make_float2(clamp_abs(a1.x, a.fp8_max), clamp_abs(a1.y, a.fp8_max));
      b0 = make_float2(clamp_abs(b0.x, a.fp8_max), clamp_abs(b0.y, a.fp8_max));
      b1 = make_float2(clamp_abs(b1.x, a.fp8_max), clamp_abs(b1.y, a.fp8_max));
    }
    ql[i / 2] = e4m3x2(a0) | (e4m3x2(a1) << 16);
    qh[i / 2] = e4m3x2(b0) | (e4m3x2(b1) << 16);
  }
  if (live) {
    // ql/qh[0..1] hold sub-chunk rev, [2..3] the other one (8 codes each)
    // One 16-byte store per half: the sub-chunk order is put back into column order first (two
    // store instructions instead of four: fewer L1 wavefronts per row, measurably faster).
    uint8_t* qrow = a.q + static_cast<int64_t>(r) * kD + 16 * j;
    const uint4 lo16 = rev ? make_uint4(ql[2], ql[3], ql[0], ql[1]) : make_uint4(ql[0], ql[1], ql[2], ql[3]);
    const uint4 hi16 = rev ? make_uint4(qh[2], qh[3], qh[0], qh[1]) : make_uint4(qh[0], qh[1], qh[2], qh[3]);
    st_stream16(qrow, lo16);
    st_stream16(qrow + 64, hi16);
    if (j == 0) a.scale[r] = sc;
  }
}

// ------------------------------------------------------------------------------ the kernel
constexpr int kReq = 2;  // cluster-launch-control requests a producer keeps in flight

// Shared memory: [pad to 1024][stages x stage_bytes][weights 2 x 128 fp32][kReq x 16-byte
// responses][full x S][empty x S][request barriers x kReq][stage start rows x S].
__host__ __device__ constexpr size_t prologue_smem_bytes(int stages, int stage_bytes) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes + 2 * kD * sizeof(float) + kReq * 16 +
         (2 * stages + kReq) * sizeof(uint64_t) + stages * sizeof(int32_t);
}

template <typename T, typename TT, int SR>
__global__ void __launch_bounds__(kThreads, 2)
    prologue_tma_kernel(const __grid_constant__ CUtensorMap xmap, const PrologueArgs a) {
  extern __shared__ unsigned char smem_raw[];
  // The 128-byte swizzle repeats every 1024 bytes: align the ring to 1024.
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int S = a.stages;
  float* wsm = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * a.stage_bytes);  // 2 x 128 floats
  uint4* resp = reinterpret_cast<uint4*>(wsm + 2 * kD);
  uint64_t* full = reinterpret_cast<uint64_t*>(resp + kReq);
  uint64_t* empty = full + S;
  uint64_t* cbar = empty + S;
  int32_t* stage_row = reinterpret_cast<int32_t*>(cbar + kReq);  // first row of each slot's chunk, -1 = end

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kTabRow = (kD / 2) * static_cast<int>(sizeof(TT));  // bytes of one table row

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps / 2);  // each stage is consumed by one half of the warps
    }
    for (int c = 0; c < kReq; ++c) mbar_init(&cbar[c], 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Programmatic dependent launch: let the next kernel in the stream start its own set-up now, and
  // wait for the previous one to finish (and its writes to be visible) before touching global memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Neither the tensor map (a kernel parameter) nor the work requests touch data the previous kernel
  // writes, so the producer lane starts both before the dependency wait.
  if (threadIdx.x == kConsumerWarps * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
    for (int c = 0; c < kReq; ++c) clc_try_cancel(&resp[c], &cbar[c]);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer (one lane)
    if (lane != 0) return;
    int k = 0;
    bool ok = true;
    int slot = 0;
    uint32_t phase = 0;  // parity of the slot's current use; its release completes phase ^ 1
    int dslot = 0;       // slot and parity of stage k - depth
    uint32_t dphase = 0;
    // Request n (n = 0, 1, ...) uses response slot n % kReq and completes that slot's barrier phase
    // n / kReq; responses are consumed in request order. The first kReq were issued above.
    int issued = kReq, answered = 0;
    uint32_t chunk = blockIdx.x;
    for (;;) {
      if (k >= S && !mbar_wait(kWaitLimitNs, &empty[slot], phase ^ 1u)) {
        ok = false;
        break;
      }
      // Keep at most `depth` stages in flight: every CTA's next stage then queues behind few
      // others, which evens out when the CTAs' data arrives.
      if (k >= a.depth) {
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
      const int32_t re = min(rs + SR, a.rows);
      const int32_t tf = static_cast<int32_t>((static_cast<uint64_t>(rs) * a.magic) >> a.shift);
      const int32_t tl = static_cast<int32_t>((static_cast<uint64_t>(re - 1) * a.magic) >> a.shift);
      const uint32_t tbytes = static_cast<uint32_t>(tl - tf + 1) * kTabRow;
      unsigned char* st = smem + static_cast<size_t>(slot) * a.stage_bytes;
      stage_row[slot] = rs;  // published to the consumers by the barrier's phase completion
      // Rows past the end of the tensor are zero-filled and still counted in full.
      mbar_arrive_expect_tx(&full[slot], 2u * half_tile<SR>() + 2u * tbytes);
      tma_load_2d(st, &xmap, 0, rs, &full[slot]);
      tma_load_2d(st + half_tile<SR>(), &xmap, kD / 2, rs, &full[slot]);
      bulk_g2s(st + 2 * half_tile<SR>(), static_cast<const unsigned char*>(a.cos) + static_cast<int64_t>(tf) * kTabRow,
               tbytes, &full[slot]);
      bulk_g2s(st + 2 * half_tile<SR>() + a.tab_block,
               static_cast<const unsigned char*>(a.sin) + static_cast<int64_t>(tf) * kTabRow, tbytes, &full[slot]);
      ++k;
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
      // The next chunk: the oldest outstanding request's answer.
      const int c = answered % kReq;
      if (!mbar_wait(kWaitLimitNs, &cbar[c], static_cast<uint32_t>(answered / kReq) & 1u)) {
        ok = false;
        break;
      }
      ++answered;
      uint32_t next;
      if (!clc_query(&resp[c], &next)) break;  // no CTA left to take over: this CTA is done
      chunk = next;
      clc_try_cancel(&resp[c], &cbar[c]);
      ++issued;
    }
    // Requests still in flight end as failures; they write this CTA's shared memory, so wait.
    while (ok && answered < issued) {
      if (!mbar_wait(kWaitLimitNs, &cbar[answered % kReq], static_cast<uint32_t>(answered / kReq) & 1u)) {
        ok = false;
        break;
      }
      ++answered;
    }
    // End marker for each consumer half (the halves take alternate stages).
    for (int e = 0; ok && e < 2; ++e) {
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
    if (!ok) {
      flag_failure(a.status);
      // Let the copies already issued land before this CTA's shared memory goes away.
      for (int j = max(0, k - S); j < k; ++j)
        if (!mbar_wait(kWaitLimitNs, &full[j % S], static_cast<uint32_t>(j / S) & 1u)) break;
      for (; answered < issued; ++answered)
        if (!mbar_wait(kWaitLimitNs, &cbar[answered % kReq], static_cast<uint32_t>(answered / kReq) & 1u)) break;
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  // Weights as fp32, permuted so that lane j's k-th float4 of a half sits at ((set*2+half)*4+k)*4+j:
  // the four lanes of a row read 64 contiguous bytes per load. Loaded while the first stages are in
  // flight; only the consumer warps synchronise on it.
  for (int i = threadIdx.x; i < 2 * kD; i += kConsumerWarps * 32) {
    const int set = i / kD, c = i % kD;
    const int half = c / 64, within = c % 64;
    const int jj = within / 16, kk = (within % 16) / 4, comp = within % 4;
    wsm[((((set * 2 + half) * 4 + kk) * 4 + jj) * 4) + comp] = Elem<T>::load1(set ? a.wk : a.wq, c);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
  const int grp = lane >> 2;  // row group within the warp
  const int j = lane & 3;     // pairs 16j..16j+15 of each half
  // A lane's 16 pairs are two sub-chunks of 8. Lanes 2 and 3 walk them in the opposite order, so
  // that in every shared-memory load the four lanes of a row touch disjoint banks (their fp32 table
  // and weight entries would otherwise sit 128 bytes apart).
  const int rev = j >> 1;
  const uint32_t wbase = smem_addr(wsm) + j * 16;
  const bool clamp = a.fp8_max != 448.0f;
  // The consumer warps work in two halves on alternate stages (even / odd), so that at any moment
  // the warps of a scheduler are at different points of their row (the serial parts -- reductions,
  // square root, reciprocals -- then overlap with the other half's arithmetic). A lane group takes
  // rows l0, l0 + 32, ... of its half's stages.
  const int half = warp / (kConsumerWarps / 2);
  const int l0 = (warp % (kConsumerWarps / 2)) * 8 + grp;

  int slot = half;  // stage k lives in slot k % S; S >= 2
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait(kWaitLimitNs, &full[slot], phase)) {
      flag_failure(a.status);
      return;
    }
    const int32_t rs = stage_row[slot];
    if (rs < 0) break;  // end marker
    const uint32_t st = smem_addr(smem + static_cast<size_t>(slot) * a.stage_bytes);
    const int32_t re = min(rs + SR, a.rows);
    const int32_t tf = static_cast<int32_t>((static_cast<uint64_t>(rs) * a.magic) >> a.shift);
#pragma unroll
    for (int u = 0; u < (SR / kGroupsPerHalf); ++u)
      prologue_row<T, TT, SR>(a, st, l0 + u * kGroupsPerHalf, j, rev, wbase, rs, re, tf, clamp);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the stage's shared memory
    slot += 2;
    if (slot >= S) {
      slot -= S;
      phase ^= 1u;
    }
  }
}

// ------------------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

namespace {

template <int SR>
bool launch_sr(const RowArgs& a, int dtype, int table_dtype, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (encode == nullptr) return false;
  const int tsz = (table_dtype == DT_FP32) ? 4 : 2;

  CUtensorMap xmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(a.rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {kD / 2, SR};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&xmap, dtype == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
             const_cast<void*>(a.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;

  PrologueArgs p{};
  p.wq = a.wq;
  p.wk = a.wk;
  p.cos = a.cos;
  p.sin = a.sin;
  p.q = a.q;
  p.scale = a.scale;
  p.status = device_status_ptr();
  p.rows = static_cast<int32_t>(a.rows);
  p.H = a.H;
  p.Hq = a.Hq;
  p.inv_h = 1.0f / static_cast<float>(a.H);
  p.eps = a.eps;
  p.fp8_max = a.fp8_max;
  p.rcp_fp8_max = static_cast<float>(1.0 / static_cast<double>(a.fp8_max));
  // r / H as (r * magic) >> shift for every r < 2^31: shift = 31 + ceil(log2 H), magic = ceil(2^shift / H).
  int lg = 0;
  while ((1LL << lg) < a.H) ++lg;
  p.shift = 31 + lg;
  p.magic = static_cast<uint64_t>(((static_cast<unsigned __int128>(1) << p.shift) + a.H - 1) / a.H);
  const int tab_rows = (SR - 1) / a.H + 2;  // tokens one stage can touch
  p.tab_block = ((tab_rows * (kD / 2) * tsz) + 127) & ~127;
  p.stage_bytes = ((2 * half_tile<SR>() + 2 * p.tab_block) + 1023) & ~1023;
  // Ring depth: as many stages (up to 12) as fit two CTAs per SM in GB300's 228 KB of shared memory.
  const int fixed = static_cast<int>(prologue_smem_bytes(12, 0));
  p.stages = (110 * 1024 - fixed) / p.stage_bytes;
  if (p.stages > 12) p.stages = 12;
  if (p.stages < 2) p.stages = 2;
  // At most 128 rows (two 64-row stages) in flight per CTA: measured best on the 4k and 32k
  // prologues. The depth must not exceed the ring: the producer waits on the full barrier of stage
  // k - depth, whose slot must not have been refilled yet.
  p.depth = 128 / SR;
  if (p.depth > p.stages) p.depth = p.stages;
  // The two consumer halves take alternate stages and wait for stage k on its slot's full barrier by
  // phase parity, which is only sound once the slot's previous use (stage k - S) has completed. With
  // S even that stage was the same half's; with S odd it was the other half's, and it has completed
  // if the producer, which issues stage j only after stage j - depth completed, keeps
  // depth <= S - 2 (the half consumed stage k - 2, issued after stage k - 2 - depth completed).
  if (p.stages % 2 != 0 && p.depth > p.stages - 2) p.depth = p.stages - 2;
  const size_t smem = prologue_smem_bytes(p.stages, p.stage_bytes);
  if (smem > 227 * 1024) return false;

  void (*kern)(const CUtensorMap, const PrologueArgs);
  if (dtype == DT_BF16)
    kern = (tsz == 4) ? prologue_tma_kernel<__nv_bfloat16, float, SR>
                      : prologue_tma_kernel<__nv_bfloat16, __nv_bfloat16, SR>;
  else
    kern = (tsz == 4) ? prologue_tma_kernel<__half, float, SR> : prologue_tma_kernel<__half, __half, SR>;
  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem)) return false;
  // One CTA per chunk of SR rows. Only the CTAs that fit on the GPU at once start; they take over
  // the rest of the grid chunk by chunk (cluster launch control), so the grid is not a wave count.
  const int grid = static_cast<int>((a.rows + SR - 1) / SR);
  // Programmatic stream serialisation: this grid may be scheduled while the previous kernel in the
  // stream drains; griddepcontrol.wait inside the kernel orders every global access after it.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, xmap, p) == cudaSuccess;
}

}  // namespace

bool launch_prologue_tma(const RowArgs& a, int dtype, int table_dtype, cudaStream_t s) {
  if (a.N != kD || a.R != kD) return false;
  if (a.rows <= 0 || a.rows > 0x7fffffffLL - 128) return false;  // row + stage size stays in int32
  if (a.token_stride != static_cast<int64_t>(a.H) * kD) return false;  // packed [T, H, 128] only
  if (a.H + 64 >= (1 << 21)) return false;
  if (!(table_dtype == DT_FP32 || table_dtype == dtype)) return false;
  if ((reinterpret_cast<uintptr_t>(a.q) & 15u) != 0) return false;
  // Short row ranges per CTA (a few stages each): 32-row stages halve the pipeline fill and drain.
  // Long ranges: 64-row stages halve the per-stage bookkeeping. Two CTAs per SM are resident.
  const int64_t rows_per_cta = a.rows / (2 * static_cast<int64_t>(sm_count()));
  if (rows_per_cta <= 1024) return launch_sr<32>(a, dtype, table_dtype, s);
  return launch_sr<64>(a, dtype, table_dtype, s);
}

}  // namespace fq
