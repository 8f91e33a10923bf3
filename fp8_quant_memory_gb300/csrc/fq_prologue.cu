// fq_prologue.cu -- the QK-Norm + RoPE + FP8 attention prologue ("case_norm_rope_quant.py" (Ch.28),
// module docstring) for head_dim 128 with the whole head rotated, as a TMA-fed persistent kernel.
//
// Data movement. The rows of the packed [T, H, 128] input are cut into chunks of SR consecutive
// (token, head) rows, one per CTA of the grid. The CTAs that are resident take over the chunks of
// CTAs that have not started yet through cluster launch control (a hardware work queue: no counter
// in global memory), so every SM keeps streaming until the last chunk is taken. One producer lane
// streams its chunks through a ring of shared-memory stages, one chunk per stage: two 2-D tensor
// TMA loads (128-byte swizzle) bring the first and second halves of the SR rows (the NeoX "lo" and
// "hi" halves) and two 1-D bulk copies bring the cos and sin rows of the tokens those rows belong
// to; an mbarrier counts the bytes. x is read from HBM once, each table row once per stage that
// needs it (L2 serves the token a stage shares with its neighbour), the two norm weights once per
// CTA straight into registers. Codes and scales go to global memory with evict-first stores.
//
// Work layout. Eight consumer warps in two halves that take alternate stages; four lanes per row,
// eight rows per warp instruction. Lane j of a row holds the NeoX pairs 16j..16j+15 of both halves,
// so every pair (p, p+64) sits in one thread and the rotation needs no data exchange. The lane keeps
// its weights -- sixteen pairs of q weights and sixteen of k weights, still packed as the 16-bit
// storage type -- in registers for the whole kernel; per row it reads its 64 bytes of x (the swizzle
// makes the eight rows of a warp instruction hit disjoint banks) and its sixteen cos and sixteen
// sin entries (lanes 2 and 3 walk their two sub-chunks of eight pairs in the opposite order, so the
// four lanes of a row read disjoint banks; the rows of a warp instruction share the token).
//
// Arithmetic (the oracle's definition with the normalisation moved past the rotation; every
// difference is a few fp32 roundings, far inside the parity tolerances -- scale within 1e-5
// relative, codes at most one step apart on at most 0.1%):
//   u = x*w, computed exactly in fp32 straight from the 16-bit operands (fma.rn.f32.bf16 / .f16:
//   two 8- or 11-bit significands); ss = sum x^2 the same way; z = rope(u): z_lo = u_lo*c - u_hi*s,
//   z_hi = u_hi*c + u_lo*s; rstd = rsqrt(ss/128 + eps) with the hardware rsqrt approximation (as
//   torch's CUDA rsqrt; ss/128 is exact as ss * 2^-7). The definition's y = rope(x*rstd*w) equals
//   rstd*z up to rounding, and |y| is largest where |z| is, so amax = max(RN(rstd * max|z|), 1e-4),
//   scale = RN(amax / fp8_max) (correctly rounded), and the codes are e4m3(RN(z * m)) with
//   m = rstd * (1/scale) (hardware reciprocal): the quotient y/scale to within a few ulps, which moves
//   a code only when it sits at an e4m3 rounding boundary.
// Signed zeros come out as in the definition (x = -0 gives the code 0x80 where y is -0): products
// keep the sign of zero, and a fused u_lo*c - u_hi*s rounds an exact zero like the unfused form.
//
// Waits are bounded: a wait that has not completed after ~1 s of %globaltimer time sets bit 0 of
// the device status word and the kernel stops issuing and consuming work (waiting, again bounded,
// for the copies and work requests it has in flight) instead of trapping.
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
constexpr int kPassRows = 32 / kLPR;                     // rows one warp instruction covers
constexpr int kConsumerWarps = 8;
constexpr int kHalfWarps = kConsumerWarps / 2;           // warps of one consumer half
constexpr int kThreads = (kConsumerWarps + 1) * 32;      // + one producer warp
constexpr int kReq = 2;                                  // work requests a producer keeps in flight

// One half of a stage's x (the NeoX lo or hi columns of SR rows, 128 bytes per row).
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
  uint32_t magic;        // t = (r * magic) >> shift == r / H for r < 2^31 (magic < 2^32 for every H)
  int32_t shift;
  int32_t rows;          // T * H
  int32_t H, Hq;
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

__device__ __forceinline__ uint4 ldg_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ uint32_t token_of(uint32_t r, uint32_t magic, int32_t shift) {
  return static_cast<uint32_t>((static_cast<uint64_t>(r) * magic) >> shift);  // one 32 x 32 -> 64 product
}

// Table entries of one sub-chunk (eight pairs) of one table row in shared memory -> 4 float2.
template <typename TT>
__device__ __forceinline__ void lds_table8(uint32_t addr, float2 (&v)[4]) {
  if constexpr (sizeof(TT) == 4) {
    const uint4 a = lds16(addr), b = lds16(addr + 16);
    v[0] = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
    v[1] = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
    v[2] = make_float2(__uint_as_float(b.x), __uint_as_float(b.y));
    v[3] = make_float2(__uint_as_float(b.z), __uint_as_float(b.w));
  } else {
    const uint4 u = lds16(addr);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = Elem<TT>::unpack(word(u, e));
  }
}

// The lane's weights of one head type in processing order: [m][0..3] the lo pairs of sub-chunk
// m ^ rev (eight 16-bit values), [m][4..7] the matching hi pairs.
struct LaneWeights {
  uint32_t v[2][8];
};

// One (token, head) row, by the four lanes of a lane group. `xrow`: the row's lo half in the stage
// (its hi half is one half tile further), `tab`: the lane's entries of the row's cos row (the sin row
// is one table block further).
template <typename T, typename TT, int SR, bool kClamp>
__device__ __forceinline__ void quant_row(const PrologueArgs& a, uint32_t xrow, int sw, int j, int rev,
                                          uint32_t tab, const LaneWeights& w, uint8_t* qrow, float* srow,
                                          bool live) {
  constexpr int kTabSub = 8 * static_cast<int>(sizeof(TT));  // bytes of one sub-chunk's table entries
  float2 zl[2][4], zh[2][4];
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
  float pm[2];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int sm = m ^ rev;  // the sub-chunk this step works on
    const uint32_t off = static_cast<uint32_t>(((2 * j + sm) ^ sw) << 4);
    const uint4 xl = lds16(xrow + off), xh = lds16(xrow + half_tile<SR>() + off);
    float2 c[4], s[4];
    lds_table8<TT>(tab + sm * kTabSub, c);
    lds_table8<TT>(tab + a.tab_block + sm * kTabSub, s);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc0 = Mixed<T>::sq_add(word(xl, e), acc0);
      acc1 = Mixed<T>::sq_add(word(xh, e), acc1);
      const float2 ul = Mixed<T>::mul(word(xl, e), w.v[m][e]);
      const float2 uh = Mixed<T>::mul(word(xh, e), w.v[m][4 + e]);
      zl[m][e] = fma2(neg2(uh), s[e], mul2(ul, c[e]));
      zh[m][e] = fma2(ul, s[e], mul2(uh, c[e]));
    }
    pm[m] = fmaxf(absmax4(absmax4(0.f, zl[m][0], zh[m][0]), zl[m][1], zh[m][1]),
                  absmax4(absmax4(0.f, zl[m][2], zh[m][2]), zl[m][3], zh[m][3]));
  }
  const float2 a01 = add2(acc0, acc1);
  float ss = a01.x + a01.y;
  float am = fmaxf(pm[0], pm[1]);
  // the row's sum of squares and max |z| over its four lanes (two interleaved chains)
#pragma unroll
  for (int o = kLPR / 2; o > 0; o >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  }
  const float rstd = rsqrtf(__fadd_rn(__fmul_rn(ss, 0.0078125f), a.eps));
  const float amax = fmaxf(__fmul_rn(rstd, am), 1e-4f);
  // scale = RN(amax / fp8_max): one product by RN(1/fp8_max) and Markstein's correction
  const float s0 = __fmul_rn(amax, a.rcp_fp8_max);
  const float sc = __fmaf_rn(__fmaf_rn(-s0, a.fp8_max, amax), a.rcp_fp8_max, s0);
  const float2 m2 = splat2(__fmul_rn(rstd, rcp_approx(sc)));
  uint32_t cl[2][2], ch[2][2];  // [step][word]: eight codes of each half per step
#pragma unroll
  for (int m = 0; m < 2; ++m) {
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      float2 l0 = mul2(zl[m][e], m2), l1 = mul2(zl[m][e + 1], m2);
      float2 h0 = mul2(zh[m][e], m2), h1 = mul2(zh[m][e + 1], m2);
      if constexpr (kClamp) {
        l0 = make_float2(clamp_abs(l0.x, a.fp8_max), clamp_abs(l0.y, a.fp8_max));
        l1 = make_float2(clamp_abs(l1.x, a.fp8_max), clamp_abs(l1.y, a.fp8_max));
        h0 = make_float2(clamp_abs(h0.x, a.fp8_max), clamp_abs(h0.y, a.fp8_max));
        h1 = make_float2(clamp_abs(h1.x, a.fp8_max), clamp_abs(h1.y, a.fp8_max));
      }
      cl[m][e / 2] = e4m3x4(l0, l1);
      ch[m][e / 2] = e4m3x4(h0, h1);
    }
  }
  if (live) {
    // one 16-byte store per half, the two steps put back into column order
    const uint4 lo16 = rev ? make_uint4(cl[1][0], cl[1][1], cl[0][0], cl[0][1])
                           : make_uint4(cl[0][0], cl[0][1], cl[1][0], cl[1][1]);
    const uint4 hi16 = rev ? make_uint4(ch[1][0], ch[1][1], ch[0][0], ch[0][1])
                           : make_uint4(ch[0][0], ch[0][1], ch[1][0], ch[1][1]);
    st_stream16(qrow, lo16);
    st_stream16(qrow + kD / 2, hi16);
    if (srow != nullptr) *srow = sc;
  }
}

// Shared memory: [pad to 1024][stages x stage_bytes][kReq x 16-byte responses][full x S][empty x S]
// [request barriers x kReq][stage start rows x S].
__host__ __device__ constexpr size_t prologue_smem_bytes(int stages, int stage_bytes) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes + kReq * 16 + (2 * stages + kReq) * sizeof(uint64_t) +
         stages * sizeof(int32_t);
}

// kUniform: every 8-row pass holds one head type (H and Hq multiples of 8: passes are 8-row aligned,
// so they never straddle a token or the q/k boundary, and a ragged stage still ends on a multiple
// of 8). The kernel then carries two copies of the row code instead of three; the smaller code
// measured 11.50 -> 11.37 us on the 4096-token workload.
template <typename T, typename TT, int SR, bool kClamp, bool kUniform>
__global__ void __launch_bounds__(kThreads, 2)
    prologue_tma_kernel(const __grid_constant__ CUtensorMap xmap, const PrologueArgs a) {
  static_assert(SR % (kHalfWarps * kPassRows) == 0, "a stage splits into whole passes per warp");
  constexpr int kWarpRows = SR / kHalfWarps;                         // consecutive rows of a stage per warp
  constexpr int kTabRow = (kD / 2) * static_cast<int>(sizeof(TT));  // bytes of one table row
  extern __shared__ unsigned char smem_raw[];
  // The 128-byte swizzle repeats every 1024 bytes: align the ring to 1024.
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int S = a.stages;
  uint4* resp = reinterpret_cast<uint4*>(smem + static_cast<size_t>(S) * a.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(resp + kReq);
  uint64_t* empty = full + S;
  uint64_t* cbar = empty + S;
  int32_t* stage_row = reinterpret_cast<int32_t*>(cbar + kReq);  // first row of each slot's chunk, -1 = end

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kHalfWarps);  // each stage is consumed by one half of the consumer warps
    }
    for (int c = 0; c < kReq; ++c) mbar_init(&cbar[c], 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Programmatic dependent launch: let the next kernel in the stream start its own set-up now, and
  // wait for the previous one to finish (and its writes to be visible) before touching global memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ClcQueue<kReq> queue;
  // Neither the tensor map (a kernel parameter) nor the work requests touch data the previous kernel
  // writes, so the producer lane starts both before the dependency wait.
  if (threadIdx.x == kConsumerWarps * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
    queue.start(resp, cbar);
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
      const uint32_t tf = token_of(static_cast<uint32_t>(rs), a.magic, a.shift);
      const uint32_t tl = token_of(static_cast<uint32_t>(re - 1), a.magic, a.shift);
      const uint32_t tbytes = (tl - tf + 1) * kTabRow;
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
      const int got = queue.next(&chunk);
      if (got < 0) ok = false;
      if (got <= 0) break;
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
      queue.drain();
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int g = lane / kLPR;  // row of the pass
  const int j = lane % kLPR;  // pairs 16j..16j+15 of each half
  // Lanes 2 and 3 walk their two sub-chunks of eight pairs in the opposite order, so that the four
  // lanes of a row read their fp32 table entries from disjoint banks.
  const int rev = j >> 1;
  // The lane's weights, packed 16-bit, in processing order.
  LaneWeights wq, wk;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int off = (16 * j + 8 * (m ^ rev)) * 2;  // bytes: eight pairs of the sub-chunk
    const unsigned char* pq = static_cast<const unsigned char*>(a.wq) + off;
    const unsigned char* pk = static_cast<const unsigned char*>(a.wk) + off;
    const uint4 ql = ldg_nc16(pq), qh = ldg_nc16(pq + kD), kl = ldg_nc16(pk), kh = ldg_nc16(pk + kD);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      wq.v[m][e] = word(ql, e);
      wq.v[m][4 + e] = word(qh, e);
      wk.v[m][e] = word(kl, e);
      wk.v[m][4 + e] = word(kh, e);
    }
  }
  const int half = warp / kHalfWarps;
  const int wrow0 = (warp % kHalfWarps) * kWarpRows + g;  // the lane group's first row of a stage
  const uint32_t tlane = static_cast<uint32_t>(j * (16 * static_cast<int>(sizeof(TT))));

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
    const uint32_t tf = token_of(static_cast<uint32_t>(rs), a.magic, a.shift);
#pragma unroll 1
    for (int p = 0; p < kWarpRows / kPassRows; ++p) {
      const int l = wrow0 + p * kPassRows;
      const int32_t r = rs + l;
      const bool live = r < re;
      const uint32_t rr = static_cast<uint32_t>(live ? r : re - 1);  // dead lanes index a live row's table
      const uint32_t t = token_of(rr, a.magic, a.shift);
      const bool isk = static_cast<int32_t>(rr - t * static_cast<uint32_t>(a.H)) >= a.Hq;
      const uint32_t xrow = st + l * 128;
      const uint32_t tab = st + 2 * half_tile<SR>() + (t - tf) * kTabRow + tlane;
      uint8_t* qrow = a.q + static_cast<int64_t>(r) * kD + 16 * j;
      float* srow = (j == 0) ? a.scale + r : nullptr;
      const int sw = l & 7;  // 128-byte swizzle phase of this row
      const uint32_t kmask = __ballot_sync(0xffffffffu, isk);
      if (kmask == 0u) {
        quant_row<T, TT, SR, kClamp>(a, xrow, sw, j, rev, tab, wq, qrow, srow, live);
      } else if (kUniform || kmask == 0xffffffffu) {
        quant_row<T, TT, SR, kClamp>(a, xrow, sw, j, rev, tab, wk, qrow, srow, live);
      } else {  // the rows of the pass mix q and k heads
        LaneWeights wsel;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int e = 0; e < 8; ++e) wsel.v[m][e] = isk ? wk.v[m][e] : wq.v[m][e];
        quant_row<T, TT, SR, kClamp>(a, xrow, sw, j, rev, tab, wsel, qrow, srow, live);
      }
    }
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

template <typename T, typename TT, int SR>
void* pick_kernel(bool clamp, bool uniform) {
  if (uniform)
    return clamp ? reinterpret_cast<void*>(prologue_tma_kernel<T, TT, SR, true, true>)
                 : reinterpret_cast<void*>(prologue_tma_kernel<T, TT, SR, false, true>);
  return clamp ? reinterpret_cast<void*>(prologue_tma_kernel<T, TT, SR, true, false>)
               : reinterpret_cast<void*>(prologue_tma_kernel<T, TT, SR, false, false>);
}

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
  p.eps = a.eps;
  p.fp8_max = a.fp8_max;
  p.rcp_fp8_max = static_cast<float>(1.0 / static_cast<double>(a.fp8_max));
  // r / H as (r * magic) >> shift for every r < 2^31: shift = 31 + ceil(log2 H), magic = ceil(2^shift / H).
  // magic < 2^shift / 2^(ceil(log2 H) - 1) = 2^32 (and 2^31 for H = 1), so it fits 32 bits.
  int lg = 0;
  while ((1LL << lg) < a.H) ++lg;
  p.shift = 31 + lg;
  const uint64_t magic = static_cast<uint64_t>(((static_cast<unsigned __int128>(1) << p.shift) + a.H - 1) / a.H);
  if (magic > 0xffffffffull) return false;
  p.magic = static_cast<uint32_t>(magic);
  const int tab_rows = (SR - 1) / a.H + 2;  // tokens one stage can touch
  p.tab_block = ((tab_rows * (kD / 2) * tsz) + 127) & ~127;
  p.stage_bytes = ((2 * half_tile<SR>() + 2 * p.tab_block) + 1023) & ~1023;
  // Ring depth: as many stages (up to 12) as fit two CTAs per SM in GB300's 228 KB of shared memory.
  const int fixed = static_cast<int>(prologue_smem_bytes(12, 0));
  p.stages = (110 * 1024 - fixed) / p.stage_bytes;
  if (p.stages > 12) p.stages = 12;
  if (p.stages < 2) p.stages = 2;
  // Rows in flight per CTA, measured: with 32-row stages (short row ranges per CTA, the 4096-token
  // workload) 128 rows 11.92 us, 256 rows 11.70 us, 384 rows 11.58 us per launch; with 64-row
  // stages (the 32768-token workload) 128 rows 130.1 us, 384 rows 132.2 us. The depth must not
  // exceed the ring: the producer waits on the full barrier of stage k - depth, whose slot must not
  // have been refilled yet.
  p.depth = (SR == 32 ? 384 : 128) / SR;
  if (p.depth > p.stages) p.depth = p.stages;
  // The two consumer halves take alternate stages and wait for stage k on its slot's full barrier by
  // phase parity, which is only sound once the slot's previous use (stage k - S) has completed. With
  // S even that stage was the same half's; with S odd it was the other half's, and it has completed
  // if the producer, which issues stage j only after stage j - depth completed, keeps
  // depth <= S - 2 (the half consumed stage k - 2, issued after stage k - 2 - depth completed).
  if (p.stages % 2 != 0 && p.depth > p.stages - 2) p.depth = p.stages - 2;
  const size_t smem = prologue_smem_bytes(p.stages, p.stage_bytes);
  if (smem > 227 * 1024) return false;

  const bool clamp = a.fp8_max != 448.0f;
  const bool uniform = a.H % 8 == 0 && a.Hq % 8 == 0;
  void* kern;
  if (dtype == DT_BF16)
    kern = (tsz == 4) ? pick_kernel<__nv_bfloat16, float, SR>(clamp, uniform)
                      : pick_kernel<__nv_bfloat16, __nv_bfloat16, SR>(clamp, uniform);
  else
    kern = (tsz == 4) ? pick_kernel<__half, float, SR>(clamp, uniform)
                      : pick_kernel<__half, __half, SR>(clamp, uniform);
  if (!ensure_dynamic_smem(kern, smem)) return false;
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
  void* args[] = {&xmap, &p};
  return cudaLaunchKernelExC(&cfg, kern, args) == cudaSuccess;
}

}  // namespace

bool launch_prologue_tma(const RowArgs& a, int dtype, int table_dtype, cudaStream_t s) {
  if (a.N != kD || a.R != kD) return false;
  if (a.rows <= 0 || a.rows > 0x7fffffffLL - 128) return false;  // row + stage size stays in int32
  if (a.token_stride != static_cast<int64_t>(a.H) * kD) return false;  // packed [T, H, 128] only
  if (!(table_dtype == DT_FP32 || table_dtype == dtype)) return false;
  if ((reinterpret_cast<uintptr_t>(a.q) & 15u) != 0) return false;
  // Short row ranges per CTA (a few stages each): 32-row stages halve the pipeline fill and drain.
  // Long ranges: 64-row stages halve the per-stage bookkeeping. Two CTAs per SM are resident.
  const int64_t rows_per_cta = a.rows / (2 * static_cast<int64_t>(sm_count()));
  if (rows_per_cta <= 1024) return launch_sr<32>(a, dtype, table_dtype, s);
  return launch_sr<64>(a, dtype, table_dtype, s);
}

}  // namespace fq
