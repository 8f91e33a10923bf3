// fq_floor.cu -- the size-matched streaming floor: a plain copy with the prologue's data movement.
//
// Not a step of the method. The QK-Norm + RoPE + FP8 prologue reads 256 bytes and writes 128 bytes
// (plus a 4-byte scale) per row; how close it gets to the HBM roofline at a given size depends as
// much on pipeline fill and drain as on bandwidth. This kernel does the least work that has the same
// traffic shape -- every 16-byte input vector read once (non-allocating load), 8 bytes written per
// vector (the XOR of its two 8-byte halves, evict-first) -- with the same work distribution (a grid of
// 512-vector chunks whose resident CTAs take over the others through cluster launch control) and
// the same programmatic dependent launch. Its time at the prologue's byte counts is the floor a
// streaming kernel of that size reaches on this GPU; the benchmark reports the prologue against it.
#include "fq_internal.h"
#include "fq_sync.cuh"

namespace fq {
namespace {

constexpr int kFloorThreads = 256;
constexpr int kFloorPer = 2;                          // vectors per thread per chunk
constexpr int kChunk = kFloorThreads * kFloorPer;     // vectors per chunk

__device__ __forceinline__ uint4 ld_nc16(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_cs8(uint2* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__global__ void __launch_bounds__(kFloorThreads) stream_floor_kernel(const uint4* __restrict__ in,
                                                                     uint2* __restrict__ out, int64_t n16,
                                                                     unsigned int* status) {
  __shared__ __align__(16) uint4 resp;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t s_next, s_ok;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint32_t chunk = blockIdx.x;
  uint32_t phase = 0;
  for (;;) {
    // Ask for the next chunk while this one streams.
    if (threadIdx.x == 0) clc_try_cancel(&resp, &bar);
    const int64_t base = static_cast<int64_t>(chunk) * kChunk + threadIdx.x;
    uint4 v[kFloorPer];
#pragma unroll
    for (int u = 0; u < kFloorPer; ++u) {
      const int64_t i = base + u * kFloorThreads;
      v[u] = i < n16 ? ld_nc16(in + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kFloorPer; ++u) {
      const int64_t i = base + u * kFloorThreads;
      if (i < n16) st_cs8(out + i, make_uint2(v[u].x ^ v[u].z, v[u].y ^ v[u].w));  // lo64 ^ hi64
    }
    if (threadIdx.x == 0) {
      uint32_t next = 0, ok = 0;
      if (mbar_wait(kWaitLimitNs, &bar, phase)) {
        ok = clc_query(&resp, &next) ? 1u : 0u;
      } else {
        flag_failure(status);
        mbar_wait(kWaitLimitNs, &bar, phase);  // the response writes shared memory: let it land
      }
      s_next = next;
      s_ok = ok;
    }
    phase ^= 1u;
    __syncthreads();
    const uint32_t ok = s_ok, next = s_next;
    __syncthreads();
    if (!ok) break;  // no CTA left to take over (or a failed wait): nothing more is requested
    chunk = next;
  }
}

}  // namespace

cudaError_t launch_stream_floor(const void* in, void* out, int64_t n16, cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>((n16 + kChunk - 1) / kChunk));
  cfg.blockDim = dim3(kFloorThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stream_floor_kernel, static_cast<const uint4*>(in), static_cast<uint2*>(out),
                            n16, device_status_ptr());
}

}  // namespace fq
