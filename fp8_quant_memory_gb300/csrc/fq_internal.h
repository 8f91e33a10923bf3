// fq_internal.h -- host-side launch interface shared by the translation units of libfq.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fq {

enum Mode : int {
  MODE_FWD = 0,         // y = dtype(x*rstd*w)
  MODE_ROPE = 1,        // y = dtype(rope(dtype(x*rstd*w)))
  MODE_ROPE_QUANT = 2,  // as MODE_ROPE, then q/scale from the rounded y; y optional
  MODE_QK = 3,          // prologue: fp32 from load to quantiser, per-head weight, per-token table
};

enum Dtype : int { DT_BF16 = 0, DT_FP16 = 1, DT_FP32 = 2 };

// One launch over `rows` rows of width N. Row r belongs to token t = r / H and head h = r % H;
// its input starts at x + t*token_stride + h*N and it uses weight (h < Hq ? wq : wk) and table
// row t. Outputs are contiguous: y/q row r at r*N, scale at r. The rmsnorm_* entry points use
// H = Hq = 1 and token_stride = N.
struct RowArgs {
  const void* x;
  const void* wq;
  const void* wk;
  const void* cos;
  const void* sin;
  void* y;         // nullable (MODE_ROPE_QUANT), unused in MODE_QK
  uint8_t* q;      // quant modes
  float* scale;    // quant modes
  int64_t rows;
  int64_t token_stride;  // elements
  int32_t H, Hq;
  int32_t N, R;
  float eps;
  float fp8_max;
  int32_t group;  // MODE_ROPE_QUANT: columns per fp32 scale, scale[r * (N / group) + g]; 0: one per row
  float* rstd;    // MODE_FWD: each row's rstd (fp32) written here when not null
  const void* bias;  // LayerNorm: the per-column bias b (nullable); wq holds the gain g
};

// Group-wise scales on the vectorised path: group % 8 == 0 and at most this many groups per row.
constexpr int kMaxVecGroups = 512;

// Vectorised path: needs N % 8 == 0, R % 16 == 0, 16-byte aligned x/w/y/cos/sin and token stride,
// 8-byte aligned q, table dtype equal to the storage dtype or fp32, and a supported width.
// Returns false (launching nothing) when the shape has no instantiation.
bool launch_rows_vector(const RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s);

// The prologue as one CTA per block of rows_per_block consecutive rows (the Ch.28 page's designs A,
// B, C), for measuring what each design moves. head_dim <= 128 fully rotated, vector layout rules.
bool launch_prologue_blocks(const RowArgs& a, int32_t rows_per_block, int dtype, int table_dtype, cudaStream_t s);

// TMA-fed persistent prologue kernel (MODE_QK, N == R == 128, 16-byte aligned token stride, table
// dtype fp32 or the storage dtype). Returns false (launching nothing) when it does not apply.
bool launch_prologue_tma(const RowArgs& a, int dtype, int table_dtype, cudaStream_t s);

// TMA-fed row-stream kernels for MODE_FWD and MODE_ROPE over contiguous rows (>= 4096 rows, the
// vectorised-path layout rules). Returns false (launching nothing) when they do not apply.
bool launch_rows_tma(const RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s);

// LayerNorm forward, y = dtype(((x - mean) * rstd) * g + b) (a.wq = g, a.bias = b or null): the TMA-fed
// wide-row kernel (>= 4096 contiguous rows, N >= 1024, vector layout) or false.
bool launch_layernorm_tma(const RowArgs& a, int dtype, cudaStream_t s);
// Every other shape: a register-resident warp-per-row kernel (N % 8 == 0, aligned, N <= 4096) or the
// scalar kernel.
void launch_layernorm(const RowArgs& a, int dtype, bool vec, cudaStream_t s);

// Scalar path: any N >= 1, even R, any alignment, any dtype combination.
void launch_rows_scalar(const RowArgs& a, int mode, int dtype, int table_dtype, cudaStream_t s);

// Backward. Partition of rows into dw chunks (depends on M only).
struct BwdPlan {
  int64_t chunks;
  int64_t rows_per_chunk;
};
BwdPlan bwd_plan(int64_t M);
size_t bwd_workspace_bytes(int64_t M, int64_t N);

struct BwdArgs {
  const void* x;
  const void* w;
  const void* g;
  void* dx;
  void* dw;
  float* dw_f32;  // nullable
  float* partial;  // [chunks, N] fp32 workspace
  const float* rstd_in;  // nullable: each row's saved rstd (used instead of recomputing it)
  int64_t M;
  int32_t N;
  float eps;
};
void launch_bwd(const BwdArgs& a, int dtype, cudaStream_t s);

// Device status word (bit 0: a bounded wait gave up). device_status_ptr() is its device address,
// passed to kernels in other translation units.
cudaError_t read_device_status(unsigned int* word, int clear, cudaStream_t s);
unsigned int* device_status_ptr();
// Launches the bounded-wait probe (one block, one wait that can only give up after limit_ms).
cudaError_t launch_wait_probe(unsigned int limit_ms, cudaStream_t s);

// The size-matched streaming floor (fq_floor.cu): n16 16-byte vectors in, 8 bytes per vector out.
cudaError_t launch_stream_floor(const void* in, void* out, int64_t n16, cudaStream_t s);

int sm_count();

// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` on the current device. The limit
// belongs to the device's context, so it is remembered per (device, kernel); thread-safe. False if
// the driver refuses.
bool ensure_dynamic_smem(const void* kernel, size_t bytes);

// Records a printf-style message for fq_last_error() on this thread and returns `code`.
int set_error(int code, const char* fmt, ...);

}  // namespace fq
