// fq_status.cu -- the device status word. Kernels that wait on something (a bounded mbarrier wait
// in a pipelined kernel) set bit 0 here instead of trapping when a wait gives up, so the context
// stays usable and the host can read the failure with fq_device_status().
#include "fq_internal.h"

namespace fq {

__device__ unsigned int g_device_status = 0u;

unsigned int* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
  return static_cast<unsigned int*>(p);
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

}  // namespace fq
