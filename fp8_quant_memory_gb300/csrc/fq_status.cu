// fq_status.cu -- the device status word. Kernels that wait on something (a bounded mbarrier wait
// in a pipelined kernel) set bit 0 here instead of trapping when a wait gives up, so the context
// stays usable and the host can read the failure with fq_device_status().
#include <map>
#include <mutex>
#include <utility>

#include "fq_internal.h"
#include "fq_sync.cuh"

namespace fq {

__device__ unsigned int g_device_status = 0u;

bool ensure_dynamic_smem(const void* kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return true;  // the default limit
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[{dev, kernel}];
  if (have >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
      cudaSuccess)
    return false;
  have = bytes;
  return true;
}

// The word's device address, looked up once per device (with that device current) and cached: in
// host code the variable's name is only a host-side stand-in. A cudaDeviceReset on a device
// invalidates the cached address (the library's device state is not rebuilt after a reset).
unsigned int* device_status_ptr() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static unsigned int* cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned int*>(p);
  }
  return cache[dev];
}

cudaError_t read_device_status(unsigned int* word, int clear, cudaStream_t s) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_device_status, sizeof(unsigned int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0u;
  e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

// One block whose only mbarrier wait can never complete (nothing arrives on the barrier): the wait
// ends by giving up after `limit_ns` and reports through the status word, the same path a stalled
// pipeline stage takes in the production kernels.
__global__ void wait_probe_kernel(unsigned int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait(limit_ns, &bar, 0u)) flag_failure(status);
  }
}

cudaError_t launch_wait_probe(unsigned int limit_ms, cudaStream_t s) {
  unsigned int* status = device_status_ptr();
  if (status == nullptr) return cudaErrorInvalidSymbol;
  wait_probe_kernel<<<1, 32, 0, s>>>(status, static_cast<uint64_t>(limit_ms) * 1000000ull);
  return cudaGetLastError();
}

}  // namespace fq
