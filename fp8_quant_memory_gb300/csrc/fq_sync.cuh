// fq_sync.cuh -- mbarrier, TMA and bulk-copy wrappers (inline PTX) shared by the pipelined kernels,
// with bounded waits: a wait that cannot complete gives up after a time limit and the kernel
// reports it through the device status word instead of hanging or trapping.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fq {

// Default limit of every pipeline wait.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; false once `limit_ns` of waiting has
// accumulated without it (or after 2^32 polls). Callers report the failure and stop; nothing traps.
// The waiting time is summed from %globaltimer readings taken every 64 polls, each step clamped to
// [0, 1 ms]: the timer can be stepped (it follows the host's clock), and a step backwards or
// forwards must neither end a healthy wait early nor stretch a failing one.
constexpr uint64_t kMaxTimerStepNs = 1000000ull;

__device__ __forceinline__ bool mbar_wait(uint64_t limit_ns, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t prev = global_ns(), waited = 0;
  for (uint32_t i = 1; i != 0; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      const uint64_t now = global_ns();
      const int64_t step = static_cast<int64_t>(now - prev);
      prev = now;
      waited += step < 0 ? 0ull : (static_cast<uint64_t>(step) > kMaxTimerStepNs ? kMaxTimerStepNs
                                                                                : static_cast<uint64_t>(step));
      if (waited > limit_ns) return false;
    }
  }
  return false;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// ------------------------------------------------------------------------------------------------
// Cluster launch control (sm_100-class): a running CTA asks the hardware scheduler to cancel the
// launch of a CTA of the same grid that has not started yet, and takes over its work. The 16-byte
// response lands in shared memory through the async proxy; completion is tracked with an mbarrier
// (16 transaction bytes), like a bulk copy. Once a CTA has observed a failed request it must not
// issue another; requests issued before that observation complete (as failures) and must still be
// waited for before the CTA exits, because they write its shared memory.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void clc_try_cancel(void* response, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, 16u);
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
          smem_addr(response)),
      "r"(smem_addr(bar))
      : "memory");
}

// Decodes a completed response: true and the cancelled CTA's blockIdx.x if the request succeeded.
__device__ __forceinline__ bool clc_query(const void* response, uint32_t* ctaid_x) {
  uint32_t ok, x = 0;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 r, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
      : "=r"(ok), "+r"(x)
      : "r"(smem_addr(response))
      : "memory");
  *ctaid_x = x;
  return ok != 0;
}

// A CTA's work queue over cluster launch control with kReq requests in flight. Request n uses
// response slot n % kReq and completes phase n / kReq of that slot's barrier; answers are read in
// issue order. The scheduler need not answer in that order: an earlier request can fail (nothing
// left to cancel) while a later one, answered first, took a CTA. So a failed answer only stops new
// requests (none may follow an observed failure); the answers still in flight are read, and a
// success among them is taken over, never dropped.
template <int kReq>
struct ClcQueue {
  uint4* resp;
  uint64_t* cbar;
  int issued;
  int answered;
  bool failed;

  __device__ __forceinline__ void start(uint4* r, uint64_t* b) {
    resp = r;
    cbar = b;
    for (int c = 0; c < kReq; ++c) clc_try_cancel(&resp[c], &cbar[c]);
    issued = kReq;
    answered = 0;
    failed = false;
  }

  // 1: a chunk to take over in *chunk (a new request replaces the answered one unless a failure was
  // seen); 0: none left and no request in flight; -1: a bounded wait gave up.
  __device__ __forceinline__ int next(uint32_t* chunk) {
    while (answered < issued) {
      const int c = answered % kReq;
      if (!mbar_wait(kWaitLimitNs, &cbar[c], static_cast<uint32_t>(answered / kReq) & 1u)) return -1;
      ++answered;
      if (clc_query(&resp[c], chunk)) {
        if (!failed) {
          clc_try_cancel(&resp[c], &cbar[c]);
          ++issued;
        }
        return 1;
      }
      failed = true;
    }
    return 0;
  }

  // After a failed wait: let the requests still in flight land (they write this CTA's shared
  // memory), each wait bounded again.
  __device__ __forceinline__ void drain() {
    for (; answered < issued; ++answered)
      if (!mbar_wait(kWaitLimitNs, &cbar[answered % kReq], static_cast<uint32_t>(answered / kReq) & 1u)) break;
  }
};

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void flag_failure(unsigned int* status) {
  if (status != nullptr) atomicOr(status, 1u);
}

}  // namespace fq
