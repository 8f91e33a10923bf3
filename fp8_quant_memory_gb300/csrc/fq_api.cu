// fq_api.cu -- the extern "C" entry points declared in include/fq.h: argument validation on the
// host (before any CUDA call), choice between the vectorised and the scalar kernels, launch, and
// error reporting through fq_last_error().
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "fq.h"
#include "fq_internal.h"

namespace {

thread_local std::string g_err;

int vfail(int code, const char* fmt, va_list ap) {
  char buf[512];
  vsnprintf(buf, sizeof(buf), fmt, ap);
  g_err = buf;
  return code;
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  const int rc = vfail(code, fmt, ap);
  va_end(ap);
  return rc;
}

int ok() {
  g_err.clear();
  return FQ_OK;
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Strict mode (fq_set_strict, or FQ_STRICT=1 in the environment at the first call): every compute
// call waits for its own stream and turns a bounded-wait failure into FQ_ERR_DEVICE.
std::atomic<int> g_strict{-1};

bool strict_mode() {
  int v = g_strict.load(std::memory_order_relaxed);
  if (v < 0) {
    const char* e = std::getenv("FQ_STRICT");
    int want = (e != nullptr && e[0] == '1') ? 1 : 0;
    g_strict.compare_exchange_strong(v, want);
    v = g_strict.load(std::memory_order_relaxed);
  }
  return v == 1;
}

int check_launch(const char* what, cudaStream_t s) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  if (strict_mode()) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    if (cap == cudaStreamCaptureStatusNone) {  // a stream being captured cannot be waited for
      unsigned int word = 0;
      e = fq::read_device_status(&word, 1, s);
      if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
      if (word & 1u)
        return fail(FQ_ERR_DEVICE, "%s: a pipelined kernel gave up on a bounded wait and skipped work", what);
    }
  }
  return ok();
}

int check_common(const char* fn, int dtype, float eps) {
  if (dtype != FQ_BF16 && dtype != FQ_FP16)
    return fail(FQ_ERR_UNSUPPORTED, "%s: dtype %d is not FQ_BF16 or FQ_FP16", fn, dtype);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(FQ_ERR_INVALID_ARG, "%s: eps must be finite and >= 0", fn);
  return FQ_OK;
}

int check_fp8_max(const char* fn, float fp8_max) {
  if (!(fp8_max > 0.0f && fp8_max <= 448.0f))
    return fail(FQ_ERR_INVALID_ARG, "%s: fp8_max must be in (0, 448], got %g", fn, static_cast<double>(fp8_max));
  return FQ_OK;
}

// `empty`: the batch has no rows, so the tables are never read and may be null.
int check_rope(const char* fn, int64_t N, int64_t R, const void* cos, const void* sin, int table_dtype,
               bool empty) {
  if (R < 0 || R % 2 != 0 || R > N)
    return fail(FQ_ERR_INVALID_ARG, "%s: rope_dim must be even and in [0, %lld], got %lld", fn,
                static_cast<long long>(N), static_cast<long long>(R));
  if (!empty && R > 0 && (cos == nullptr || sin == nullptr))
    return fail(FQ_ERR_INVALID_ARG, "%s: cos/sin are null", fn);
  if (table_dtype != FQ_BF16 && table_dtype != FQ_FP16 && table_dtype != FQ_FP32)
    return fail(FQ_ERR_UNSUPPORTED, "%s: table dtype %d is not FQ_BF16, FQ_FP16 or FQ_FP32", fn, table_dtype);
  return FQ_OK;
}

// Rows are indexed with 32-bit integers inside the kernels; element offsets are 64-bit.
constexpr int64_t kMaxRows = 0x7fffffffLL;
constexpr int64_t kMaxWidth = 1LL << 24;

bool env_is(const char* name, const char* value) {
  const char* v = std::getenv(name);
  return v != nullptr && std::string(v) == value;
}

// Launch a row problem on the vectorised kernel when layout permits, else on the scalar kernel.
int launch_rows(const char* fn, const fq::RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s) {
  cudaGetLastError();  // drop a stale non-sticky error from an unrelated earlier call
  const int64_t tsize = (table_dtype == FQ_FP32) ? 4 : 2;
  bool vec = (a.N % 8 == 0) && (a.R % 16 == 0) && aligned(a.x, 16) && aligned(a.wq, 16) &&
             aligned(a.wk, 16) && (a.token_stride * 2) % 16 == 0;
  if (a.R > 0) vec = vec && aligned(a.cos, 16) && aligned(a.sin, 16) && ((a.R / 2) * tsize) % 16 == 0;
  if (a.y != nullptr) vec = vec && aligned(a.y, 16);
  if (a.q != nullptr) vec = vec && aligned(a.q, 8);
  if (a.scale != nullptr) vec = vec && aligned(a.scale, 4);
  if (a.group > 0) vec = vec && (a.group % 8 == 0) && (a.N / a.group) <= fq::kMaxVecGroups;
  // FQ_PROLOGUE_KERNEL=generic (prologue) and FQ_ROWS_KERNEL=generic (RMSNorm forward, RMSNorm +
  // RoPE) select the generic vectorised kernel instead of the TMA-fed one (diagnostic switches: both
  // compute the same result).
  if (vec && mode == fq::MODE_QK && !env_is("FQ_PROLOGUE_KERNEL", "generic") &&
      fq::launch_prologue_tma(a, dtype, table_dtype, s))
    return check_launch(fn, s);
  if (vec && (mode == fq::MODE_FWD || mode == fq::MODE_ROPE || mode == fq::MODE_ROPE_QUANT) &&
      !env_is("FQ_ROWS_KERNEL", "generic") &&
      fq::launch_rows_tma(a, mode, dtype, table_dtype, s))
    return check_launch(fn, s);
  if (!(vec && fq::launch_rows_vector(a, mode, dtype, table_dtype, s)))
    fq::launch_rows_scalar(a, mode, dtype, table_dtype, s);
  return check_launch(fn, s);
}

}  // namespace

namespace fq {

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  const int rc = vfail(code, fmt, ap);
  va_end(ap);
  return rc;
}

int sm_count() {
  static int cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace fq

extern "C" {

const char* fq_last_error(void) { return g_err.c_str(); }

int fq_version(void) { return 2; }

int fq_device_status(unsigned int* word, int clear, cudaStream_t stream) {
  if (word == nullptr) return fail(FQ_ERR_INVALID_ARG, "fq_device_status: word is null");
  const cudaError_t e = fq::read_device_status(word, clear, stream);
  if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "fq_device_status: %s", cudaGetErrorString(e));
  return ok();
}

int fq_check_bounded_wait(unsigned int limit_ms, cudaStream_t stream) {
  if (limit_ms < 1 || limit_ms > 10000)
    return fail(FQ_ERR_INVALID_ARG, "fq_check_bounded_wait: limit_ms must be in [1, 10000], got %u", limit_ms);
  cudaGetLastError();
  const cudaError_t e = fq::launch_wait_probe(limit_ms, stream);
  if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "fq_check_bounded_wait: %s", cudaGetErrorString(e));
  return ok();
}

int fq_set_strict(int on) {
  const int prev = strict_mode() ? 1 : 0;
  g_strict.store(on ? 1 : 0, std::memory_order_relaxed);
  return prev;
}

int fq_stream_floor(const void* in, void* out, int64_t n16, cudaStream_t stream) {
  if (n16 < 0 || n16 > (static_cast<int64_t>(1) << 40))
    return fail(FQ_ERR_INVALID_ARG, "fq_stream_floor: need 0 <= n16 <= 2^40, got %lld", static_cast<long long>(n16));
  if (n16 == 0) return ok();
  if (in == nullptr || out == nullptr) return fail(FQ_ERR_INVALID_ARG, "fq_stream_floor: null pointer");
  if (!aligned(in, 16) || !aligned(out, 8))
    return fail(FQ_ERR_INVALID_ARG, "fq_stream_floor: in must be 16-byte and out 8-byte aligned");
  cudaGetLastError();
  const cudaError_t e = fq::launch_stream_floor(in, out, n16, stream);
  if (e != cudaSuccess) return fail(FQ_ERR_CUDA, "fq_stream_floor: %s", cudaGetErrorString(e));
  return ok();
}

int fq_rmsnorm_fwd_rstd(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N, int dtype,
                        float eps, cudaStream_t stream) {
  const char* fn = rstd != nullptr ? "fq_rmsnorm_fwd_rstd" : "fq_rmsnorm_fwd";
  if (int rc = check_common(fn, dtype, eps)) return rc;
  if (M < 0 || N < 1 || M > kMaxRows || N > kMaxWidth)
    return fail(FQ_ERR_INVALID_ARG, "%s: need 0 <= M <= 2^31-1 and 1 <= N <= 2^24", fn);
  if (M == 0) return ok();
  if (x == nullptr || w == nullptr || y == nullptr) return fail(FQ_ERR_INVALID_ARG, "%s: null pointer", fn);
  fq::RowArgs a{};
  a.x = x;
  a.wq = a.wk = w;
  a.y = y;
  a.rstd = rstd;
  a.rows = M;
  a.token_stride = N;
  a.H = a.Hq = 1;
  a.N = static_cast<int32_t>(N);
  a.R = 0;
  a.eps = eps;
  a.fp8_max = 448.0f;
  return launch_rows(fn, a, fq::MODE_FWD, dtype, dtype, stream);
}

int fq_layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y, int64_t M, int64_t N, int dtype,
                     float eps, cudaStream_t stream) {
  const char* fn = "fq_layernorm_fwd";
  if (int rc = check_common(fn, dtype, eps)) return rc;
  if (M < 0 || N < 1 || M > kMaxRows || N > kMaxWidth)
    return fail(FQ_ERR_INVALID_ARG, "%s: need 0 <= M <= 2^31-1 and 1 <= N <= 2^24", fn);
  if (M == 0) return ok();
  if (x == nullptr || gamma == nullptr || y == nullptr) return fail(FQ_ERR_INVALID_ARG, "%s: null pointer", fn);
  cudaGetLastError();
  fq::RowArgs a{};
  a.x = x;
  a.wq = a.wk = gamma;
  a.bias = beta;
  a.y = y;
  a.rows = M;
  a.token_stride = N;
  a.H = a.Hq = 1;
  a.N = static_cast<int32_t>(N);
  a.eps = eps;
  a.fp8_max = 448.0f;
  const bool vec = (N % 8 == 0) && aligned(x, 16) && aligned(gamma, 16) && aligned(y, 16) &&
                   (beta == nullptr || aligned(beta, 16));
  fq::launch_layernorm(a, dtype, vec, stream);
  return check_launch(fn, stream);
}

int fq_rmsnorm_fwd(const void* x, const void* w, void* y, int64_t M, int64_t N, int dtype, float eps,
                   cudaStream_t stream) {
  return fq_rmsnorm_fwd_rstd(x, w, y, nullptr, M, N, dtype, eps, stream);
}

int fq_rmsnorm_rope(const void* x, const void* w, const void* cos, const void* sin, void* y, int64_t M,
                    int64_t N, int64_t rope_dim, int dtype, int table_dtype, float eps,
                    cudaStream_t stream) {
  const char* fn = "fq_rmsnorm_rope";
  if (int rc = check_common(fn, dtype, eps)) return rc;
  if (M < 0 || N < 1 || M > kMaxRows || N > kMaxWidth)
    return fail(FQ_ERR_INVALID_ARG, "%s: need 0 <= M <= 2^31-1 and 1 <= N <= 2^24", fn);
  if (int rc = check_rope(fn, N, rope_dim, cos, sin, table_dtype, M == 0)) return rc;
  if (M == 0) return ok();
  if (x == nullptr || w == nullptr || y == nullptr) return fail(FQ_ERR_INVALID_ARG, "%s: null pointer", fn);
  fq::RowArgs a{};
  a.x = x;
  a.wq = a.wk = w;
  a.cos = cos;
  a.sin = sin;
  a.y = y;
  a.rows = M;
  a.token_stride = N;
  a.H = a.Hq = 1;
  a.N = static_cast<int32_t>(N);
  a.R = static_cast<int32_t>(rope_dim);
  a.eps = eps;
  a.fp8_max = 448.0f;
  return launch_rows(fn, a, fq::MODE_ROPE, dtype, table_dtype, stream);
}

}  // extern "C"

namespace {

// Shared body of fq_rmsnorm_rope_quant (group = 0: one scale per row) and
// fq_rmsnorm_rope_quant_groups (group = columns per scale).
int rope_quant(const char* fn, const void* x, const void* w, const void* cos, const void* sin, void* y, uint8_t* q,
               float* scale, int64_t M, int64_t N, int64_t rope_dim, int64_t group, int dtype, int table_dtype,
               float eps, float fp8_max, cudaStream_t stream) {
  if (int rc = check_common(fn, dtype, eps)) return rc;
  if (int rc = check_fp8_max(fn, fp8_max)) return rc;
  if (M < 0 || N < 1 || M > kMaxRows || N > kMaxWidth)
    return fail(FQ_ERR_INVALID_ARG, "%s: need 0 <= M <= 2^31-1 and 1 <= N <= 2^24", fn);
  if (group < 0 || (group > 0 && N % group != 0))
    return fail(FQ_ERR_INVALID_ARG, "%s: group_size must divide N (N = %lld, group_size = %lld)", fn,
                static_cast<long long>(N), static_cast<long long>(group));
  if (int rc = check_rope(fn, N, rope_dim, cos, sin, table_dtype, M == 0)) return rc;
  if (M == 0) return ok();
  if (x == nullptr || w == nullptr || q == nullptr || scale == nullptr)
    return fail(FQ_ERR_INVALID_ARG, "%s: null pointer", fn);
  fq::RowArgs a{};
  a.x = x;
  a.wq = a.wk = w;
  a.cos = cos;
  a.sin = sin;
  a.y = y;
  a.q = q;
  a.scale = scale;
  a.rows = M;
  a.token_stride = N;
  a.H = a.Hq = 1;
  a.N = static_cast<int32_t>(N);
  a.R = static_cast<int32_t>(rope_dim);
  a.eps = eps;
  a.fp8_max = fp8_max;
  a.group = (group == N) ? 0 : static_cast<int32_t>(group);  // one group per row is the per-row path
  return launch_rows(fn, a, fq::MODE_ROPE_QUANT, dtype, table_dtype, stream);
}

}  // namespace

extern "C" {

int fq_rmsnorm_rope_quant(const void* x, const void* w, const void* cos, const void* sin, void* y,
                          uint8_t* q, float* scale, int64_t M, int64_t N, int64_t rope_dim, int dtype,
                          int table_dtype, float eps, float fp8_max, cudaStream_t stream) {
  return rope_quant("fq_rmsnorm_rope_quant", x, w, cos, sin, y, q, scale, M, N, rope_dim, 0, dtype, table_dtype,
                    eps, fp8_max, stream);
}

int fq_rmsnorm_rope_quant_groups(const void* x, const void* w, const void* cos, const void* sin, void* y,
                                 uint8_t* q, float* scale, int64_t M, int64_t N, int64_t rope_dim,
                                 int64_t group_size, int dtype, int table_dtype, float eps, float fp8_max,
                                 cudaStream_t stream) {
  if (group_size < 1)
    return fail(FQ_ERR_INVALID_ARG, "fq_rmsnorm_rope_quant_groups: group_size must be >= 1, got %lld",
                static_cast<long long>(group_size));
  return rope_quant("fq_rmsnorm_rope_quant_groups", x, w, cos, sin, y, q, scale, M, N, rope_dim, group_size, dtype,
                    table_dtype, eps, fp8_max, stream);
}

}  // extern "C"

namespace {

// Validation and argument packing shared by the prologue entry points; returns FQ_OK and fills `a`
// (a.rows == 0: nothing to launch).
int prologue_args(const char* fn, const void* qk, int64_t token_stride, const void* wq, const void* wk,
                  const void* cos, const void* sin, uint8_t* q_out, float* scale, int64_t T, int64_t Hq,
                  int64_t Hk, int64_t D, int64_t rope_dim, int dtype, int table_dtype, float eps, float fp8_max,
                  fq::RowArgs* a) {
  if (int rc = check_common(fn, dtype, eps)) return rc;
  if (int rc = check_fp8_max(fn, fp8_max)) return rc;
  if (T < 0 || Hq < 0 || Hk < 0 || Hq + Hk < 1 || D < 1 || D > kMaxWidth || Hq + Hk > kMaxWidth)
    return fail(FQ_ERR_INVALID_ARG, "%s: need T >= 0, Hq, Hk >= 0, Hq + Hk >= 1, D >= 1", fn);
  const int64_t H = Hq + Hk;
  if (token_stride < H * D)
    return fail(FQ_ERR_INVALID_ARG, "%s: token_stride %lld < (Hq+Hk)*D = %lld", fn,
                static_cast<long long>(token_stride), static_cast<long long>(H * D));
  if (T > kMaxRows / H) return fail(FQ_ERR_INVALID_ARG, "%s: T*(Hq+Hk) must be < 2^31", fn);
  if (int rc = check_rope(fn, D, rope_dim, cos, sin, table_dtype, T == 0)) return rc;
  *a = fq::RowArgs{};
  if (T == 0) return ok();
  if (qk == nullptr || wq == nullptr || wk == nullptr || q_out == nullptr || scale == nullptr)
    return fail(FQ_ERR_INVALID_ARG, "%s: null pointer", fn);
  a->x = qk;
  a->wq = wq;
  a->wk = wk;
  a->cos = cos;
  a->sin = sin;
  a->y = nullptr;
  a->q = q_out;
  a->scale = scale;
  a->rows = T * H;
  a->token_stride = token_stride;
  a->H = static_cast<int32_t>(H);
  a->Hq = static_cast<int32_t>(Hq);
  a->N = static_cast<int32_t>(D);
  a->R = static_cast<int32_t>(rope_dim);
  a->eps = eps;
  a->fp8_max = fp8_max;
  return FQ_OK;
}

}  // namespace

extern "C" {

int fq_qk_norm_rope_quant(const void* qk, int64_t token_stride, const void* wq, const void* wk,
                          const void* cos, const void* sin, uint8_t* q_out, float* scale, int64_t T,
                          int64_t Hq, int64_t Hk, int64_t D, int64_t rope_dim, int dtype,
                          int table_dtype, float eps, float fp8_max, cudaStream_t stream) {
  const char* fn = "fq_qk_norm_rope_quant";
  fq::RowArgs a;
  if (int rc = prologue_args(fn, qk, token_stride, wq, wk, cos, sin, q_out, scale, T, Hq, Hk, D, rope_dim, dtype,
                             table_dtype, eps, fp8_max, &a))
    return rc;
  if (a.rows == 0) return ok();
  return launch_rows(fn, a, fq::MODE_QK, dtype, table_dtype, stream);
}

int fq_qk_norm_rope_quant_blocks(const void* qk, int64_t token_stride, const void* wq, const void* wk,
                                 const void* cos, const void* sin, uint8_t* q_out, float* scale, int64_t T,
                                 int64_t Hq, int64_t Hk, int64_t D, int64_t rope_dim, int64_t rows_per_block,
                                 int dtype, int table_dtype, float eps, float fp8_max, cudaStream_t stream) {
  const char* fn = "fq_qk_norm_rope_quant_blocks";
  if (rows_per_block < 1 || rows_per_block > 128)
    return fail(FQ_ERR_INVALID_ARG, "%s: rows_per_block must be in [1, 128], got %lld", fn,
                static_cast<long long>(rows_per_block));
  fq::RowArgs a;
  if (int rc = prologue_args(fn, qk, token_stride, wq, wk, cos, sin, q_out, scale, T, Hq, Hk, D, rope_dim, dtype,
                             table_dtype, eps, fp8_max, &a))
    return rc;
  if (a.rows == 0) return ok();
  const int64_t tsize = (table_dtype == FQ_FP32) ? 4 : 2;
  const bool vec = D == rope_dim && D % 16 == 0 && D <= 128 && aligned(qk, 16) && aligned(wq, 16) &&
                   aligned(wk, 16) && aligned(cos, 16) && aligned(sin, 16) && (token_stride * 2) % 16 == 0 &&
                   ((rope_dim / 2) * tsize) % 16 == 0 && aligned(q_out, 8) && aligned(scale, 4);
  cudaGetLastError();
  if (!vec || !fq::launch_prologue_blocks(a, static_cast<int32_t>(rows_per_block), dtype, table_dtype, stream))
    return fail(FQ_ERR_UNSUPPORTED,
                "%s: needs head_dim = rope_dim <= 128, a multiple of 16, and 16-byte aligned tensors", fn);
  return check_launch(fn, stream);
}
size_t fq_rmsnorm_bwd_workspace_bytes(int64_t M, int64_t N) {
  if (M <= 0 || N <= 0) return 0;
  return fq::bwd_workspace_bytes(M, N);
}

}  // extern "C"

namespace {

int rmsnorm_bwd(const char* fn, const void* x, const void* w, const void* grad_y, const float* rstd, void* dx,
                void* dw, float* dw_f32, void* workspace, size_t workspace_bytes, int64_t M, int64_t N, int dtype,
                float eps, cudaStream_t stream) {
  if (int rc = check_common(fn, dtype, eps)) return rc;
  if (M < 0 || N < 1 || M > kMaxRows || N > kMaxWidth)
    return fail(FQ_ERR_INVALID_ARG, "%s: need 0 <= M <= 2^31-1 and 1 <= N <= 2^24", fn);
  if (w == nullptr || dw == nullptr || (M > 0 && (x == nullptr || grad_y == nullptr || dx == nullptr)))
    return fail(FQ_ERR_INVALID_ARG, "%s: null pointer", fn);
  const size_t need = fq_rmsnorm_bwd_workspace_bytes(M, N);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need))
    return fail(FQ_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
  if (need > 0 && !aligned(workspace, 16)) return fail(FQ_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", fn);
  cudaGetLastError();
  fq::BwdArgs a{};
  a.x = x;
  a.w = w;
  a.g = grad_y;
  a.dx = dx;
  a.dw = dw;
  a.dw_f32 = dw_f32;
  a.partial = static_cast<float*>(workspace);
  a.rstd_in = rstd;
  a.M = M;
  a.N = static_cast<int32_t>(N);
  a.eps = eps;
  fq::launch_bwd(a, dtype, stream);
  return check_launch(fn, stream);
}

}  // namespace

extern "C" {

int fq_rmsnorm_bwd(const void* x, const void* w, const void* grad_y, void* dx, void* dw, float* dw_f32,
                   void* workspace, size_t workspace_bytes, int64_t M, int64_t N, int dtype, float eps,
                   cudaStream_t stream) {
  return rmsnorm_bwd("fq_rmsnorm_bwd", x, w, grad_y, nullptr, dx, dw, dw_f32, workspace, workspace_bytes, M, N, dtype,
                     eps, stream);
}

int fq_rmsnorm_bwd_rstd(const void* x, const void* w, const void* grad_y, const float* rstd, void* dx, void* dw,
                        float* dw_f32, void* workspace, size_t workspace_bytes, int64_t M, int64_t N, int dtype,
                        cudaStream_t stream) {
  if (rstd == nullptr && M > 0) return fail(FQ_ERR_INVALID_ARG, "fq_rmsnorm_bwd_rstd: rstd is null");
  return rmsnorm_bwd("fq_rmsnorm_bwd_rstd", x, w, grad_y, rstd, dx, dw, dw_f32, workspace, workspace_bytes, M, N,
                     dtype, 0.0f, stream);
}


}  // extern "C"
