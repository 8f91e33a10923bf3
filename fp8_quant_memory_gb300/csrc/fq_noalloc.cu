// fq_noalloc.cu -- RMSNorm backward for callers that cannot allocate device memory.
//
// fq_rmsnorm_bwd needs a caller-provided workspace for the fp32 per-chunk partial column sums of dw.
// Some callers have no way to provide one: a plugin loaded into a host framework that owns every
// device buffer through its own pool and hands the plugin only its tensors, or a latency-critical
// loop that must never call cudaMalloc (which can synchronise the whole device). This entry point
// takes the same inputs and outputs but keeps the partial sums in a fixed-size array that lives in
// the library's own device memory: every GPU that loads the library holds it until the process
// exits. Nothing here calls cudaMalloc, cudaFree or any other allocating routine.
#include <mutex>

#include "fq.h"
#include "fq_internal.h"

namespace {

constexpr size_t kScratchBytes = FQ_NOALLOC_SCRATCH_BYTES;

// The scratch: fp32 partial column sums, [chunks, N]. Stage 1 overwrites every element it later
// reads, so nothing has to be cleared between calls; it keeps the last call's contents.
static __device__ __align__(256) float g_bwd_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device. In host code the array's name is only a
// host-side stand-in, so the address is looked up once per device (with that device current) and
// cached.
cudaError_t scratch_on_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int fq_rmsnorm_bwd_noalloc(const void* x, const void* w, const void* grad_y, void* dx, void* dw,
                                      float* dw_f32, int64_t M, int64_t N, int dtype, float eps,
                                      cudaStream_t stream) {
  const size_t need = fq_rmsnorm_bwd_workspace_bytes(M, N);
  if (need > kScratchBytes)
    return fq::set_error(FQ_ERR_INVALID_ARG,
                         "fq_rmsnorm_bwd_noalloc: an [%lld, %lld] problem needs %zu bytes of scratch, the "
                         "built-in scratch holds %zu; use fq_rmsnorm_bwd with a workspace",
                         static_cast<long long>(M), static_cast<long long>(N), need, kScratchBytes);
  float* scratch = nullptr;
  if (need > 0) {
    const cudaError_t e = scratch_on_current_device(&scratch);
    if (e != cudaSuccess)
      return fq::set_error(FQ_ERR_CUDA, "fq_rmsnorm_bwd_noalloc: scratch address lookup failed: %s",
                           cudaGetErrorString(e));
  }
  // Same validation, kernels and reduction order as the workspace entry point.
  return fq_rmsnorm_bwd(x, w, grad_y, dx, dw, dw_f32, scratch, need > 0 ? kScratchBytes : 0, M, N, dtype, eps,
                        stream);
}
