/*
 * fq.h -- C ABI of libfq: fused RMSNorm -> NeoX partial RoPE -> per-row FP8 (e4m3fn) quantisation
 * on GB300 (sm_103a), plus the standalone RMSNorm forward and backward.
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller. The library never allocates,
 *     frees or retains any of them; it does not keep pointers past the call.
 *   - Work is enqueued on `stream` (0 = the legacy default stream) and runs asynchronously: outputs
 *     are valid once the stream reaches that point. No entry point synchronises.
 *   - Shapes are element counts. All tensors are row-major and contiguous unless a stride argument
 *     says otherwise. Output buffers must not overlap input buffers.
 *   - Storage dtypes: FQ_BF16 (bfloat16) or FQ_FP16 (IEEE binary16) for x, w, y, grad_y, dx, dw.
 *     Rotary tables: FQ_BF16, FQ_FP16 or FQ_FP32. FP8 outputs are uint8 codes in OCP E4M3 "fn"
 *     encoding (bias 7, max +-448, no infinities, NaN = S.1111.111).
 *   - Return value: FQ_OK, or an fq_status error code. On error nothing was launched and a
 *     message is available from fq_last_error() (per thread). Argument checks happen on the host
 *     before any CUDA call, so an invalid call never touches the device.
 *   - Rows of 16-byte aligned, 8-element multiples take the vectorised kernels; anything else
 *     (odd widths, unaligned pointers, rope_dim not a multiple of 16, other table dtypes) takes a
 *     scalar kernel with the same results. No combination falls back to the host.
 *
 * Sources of the definitions (tutorial pages, cited by title and function):
 *   "rmsnorm_rope_quant.py" (Ch.13 operators I, fusion capstone): torch_reference_fused,
 *       _torch_rope_neox, rms_norm_rope_fused, rms_norm_rope_quant_fused.
 *   "rmsnorm_tl.py" (Ch.17 end-to-end training): _rmsnorm_fwd, RMSNormTileLang.backward.
 *   "case_norm_rope_quant.py" (Ch.28 operator design methodology): the QK-Norm + RoPE + FP8
 *       attention prologue (module docstring) and design C (one token's rows share the lookups).
 */
#ifndef FQ_H_
#define FQ_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum fq_status {
  FQ_OK = 0,
  FQ_ERR_INVALID_ARG = 1, /* null pointer, non-positive or inconsistent shape, odd rope_dim,
                             rope_dim > row width, fp8_max outside (0, 448], eps < 0 or not finite */
  FQ_ERR_UNSUPPORTED = 2, /* dtype code not accepted by this entry point */
  FQ_ERR_MISALIGNED = 3,  /* reserved: misaligned inputs take the scalar path instead */
  FQ_ERR_CUDA = 4,        /* a CUDA call failed (launch error, no device); see fq_last_error() */
  FQ_ERR_DEVICE = 5       /* strict mode only (fq_set_strict): a kernel reported a failure through the
                             device status word */
};

/* Storage dtype codes. */
enum fq_dtype { FQ_BF16 = 0, FQ_FP16 = 1, FQ_FP32 = 2 };

/* Message describing the last error returned on the calling thread ("" if none). The string is
 * owned by the library and stays valid until the next call on the same thread. */
const char* fq_last_error(void);

/* Library ABI version (incremented on any signature change). */
int fq_version(void);

/* Reads the device status word of the current device after synchronising `stream`, optionally
 * clearing it. Bit 0 (value 1): a pipelined kernel gave up on a bounded wait and skipped its
 * remaining work. `*word` receives the bits. Returns FQ_OK or FQ_ERR_CUDA.
 * Compute calls return as soon as their work is enqueued, before a kernel can have given up on a
 * wait, so a plain FQ_OK does not say that the work completed: either read this word after the
 * stream reaches the call, or turn on strict mode (fq_set_strict). The word is one per device and
 * shared by every stream and call. The library looks up its device address once per device; after
 * a cudaDeviceReset on that device the library must not be used there again in the same process. */
int fq_device_status(unsigned int* word, int clear, cudaStream_t stream);

/* Strict mode on (1) or off (0); returns the previous setting. Also turned on by FQ_STRICT=1 in the
 * environment at the first call. In strict mode every compute entry point, after enqueuing its work,
 * synchronises its stream, reads and clears the device status word, and returns FQ_ERR_DEVICE if bit
 * 0 was set -- attributing to this call any bounded-wait failure since the word was last cleared.
 * While `stream` is being captured into a CUDA graph it cannot be waited for, and strict mode
 * checks nothing. Strict mode trades the asynchronous launch for an immediate answer (a debugging
 * and validation mode). The tutorial pages have no counterpart. */
int fq_set_strict(int on);

/* Diagnostic for the bounded waits of the pipelined kernels: enqueues one block whose single
 * mbarrier wait can never complete (nothing arrives on the barrier). The wait gives up after
 * limit_ms milliseconds (1..10000) and sets bit 0 of the device status word -- the path a stalled
 * pipeline stage takes -- instead of hanging or trapping; the context stays usable. After the
 * stream reaches it, fq_device_status reports bit 0 set. Returns FQ_OK, FQ_ERR_INVALID_ARG or
 * FQ_ERR_CUDA. The tutorial pages have no counterpart (they have no pipelined kernel). */
int fq_check_bounded_wait(unsigned int limit_ms, cudaStream_t stream);

/* Measurement aid, not a step of the method: the size-matched streaming floor. Reads n16 16-byte
 * vectors from `in` (device, 16-byte aligned) once each and writes 8 bytes per vector to `out`
 * (device, 8-byte aligned, n16 * 8 bytes): out[i] = (low 8 bytes of in[i]) XOR (high 8 bytes of
 * in[i]), i.e. 32-bit word k of out[i] is word k XOR word k + 2 of in[i]. That is the traffic shape of the
 * QK-norm prologue ("case_norm_rope_quant.py" (Ch.28), `Design.payload_bytes`: 2 bytes read and 1
 * written per element) with no arithmetic, the same work distribution (cluster launch control over
 * 512-vector chunks) and the same programmatic dependent launch, so its time at the prologue's byte
 * counts is what a streaming kernel of that size reaches on the GPU. 0 <= n16 <= 2^40 (n16 = 0 is a
 * no-op). Caller-owned memory, asynchronous on `stream`. Returns FQ_OK, FQ_ERR_INVALID_ARG (null,
 * misaligned, out of range) or FQ_ERR_CUDA. */
int fq_stream_floor(const void* in, void* out, int64_t n16, cudaStream_t stream);

/*
 * RMSNorm forward ("rmsnorm_tl.py", _rmsnorm_fwd):
 *   rstd_i = 1 / sqrt(sum_j x_ij^2 / N + eps)   (fp32)
 *   y_ij   = dtype((x_ij * rstd_i) * w_j)        (fp32 products, one rounding to dtype)
 * x, y: [M, N] dtype; w: [N] dtype. M >= 0 (M = 0 is a no-op), N >= 1.
 */
int fq_rmsnorm_fwd(const void* x, const void* w, void* y, int64_t M, int64_t N, int dtype, float eps,
                   cudaStream_t stream);

/*
 * RMSNorm forward that also saves each row's rstd for the backward (the alternative to the Ch.17
 * page's RMSNormTileLang, which saves only x and w and recomputes rstd in backward):
 *   y as fq_rmsnorm_fwd;  rstd[i] = 1 / sqrt(sum_j x_ij^2 / N + eps)   (fp32, [M])
 * rstd may be null (then this is fq_rmsnorm_fwd). Other arguments and errors as fq_rmsnorm_fwd.
 */
int fq_rmsnorm_fwd_rstd(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N, int dtype,
                        float eps, cudaStream_t stream);

/*
 * LayerNorm forward, the fused kernel of "ledger.py" (Ch.13 ledger, layer_norm:
 * y = (x - mean) / sqrt(var + eps) * g + b, one read of x, g, b and one write of y):
 *   mean_i = sum_j x_ij / N;  var_i = sum_j (x_ij - mean_i)^2 / N;  rstd_i = 1/sqrt(var_i + eps) (fp32)
 *   y_ij   = dtype(((x_ij - mean_i) * rstd_i) * gamma_j + beta_j)     (each fp32 step rounded)
 * x, y: [M, N] dtype; gamma: [N] dtype; beta: [N] dtype or null (no bias). M >= 0 (0: no-op), N >= 1.
 * The page gives the formula only (a byte ledger); the cast points follow the RMSNorm definitions.
 */
int fq_layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y, int64_t M, int64_t N, int dtype,
                     float eps, cudaStream_t stream);

/*
 * RMSNorm + NeoX partial RoPE ("rmsnorm_rope_quant.py", rms_norm_rope_fused and the first two
 * steps of torch_reference_fused):
 *   normed_ij = dtype((x_ij * rstd_i) * w_j)
 *   for p < R/2, lo = normed[i, N-R+p], hi = normed[i, N-R+R/2+p], c = cos[i,p], s = sin[i,p]:
 *     y[i, N-R+p]     = dtype(lo*c - hi*s)
 *     y[i, N-R+R/2+p] = dtype(hi*c + lo*s)
 *   the first N-R columns of y are normed unchanged.
 * x, y: [M, N] dtype; w: [N]; cos, sin: [M, R/2] table_dtype (one table row per x row).
 * R = rope_dim: even, 0 <= R <= N (R = 0: no rotation; cos/sin may then be null).
 */
int fq_rmsnorm_rope(const void* x, const void* w, const void* cos, const void* sin, void* y, int64_t M,
                    int64_t N, int64_t rope_dim, int dtype, int table_dtype, float eps,
                    cudaStream_t stream);

/*
 * RMSNorm + NeoX partial RoPE + per-row FP8 ("rmsnorm_rope_quant.py", torch_reference_fused):
 *   y as in fq_rmsnorm_rope (rounded to dtype);
 *   scale_i = max(max_j |y_ij|, 1e-4) / fp8_max                       (fp32)
 *   q_ij    = e4m3fn_round_to_nearest_even(clamp(y_ij / scale_i, -fp8_max, fp8_max))
 * y: [M, N] dtype, or null to skip writing it (q and scale are unchanged by that choice);
 * q: [M, N] uint8 e4m3fn codes; scale: [M] fp32. fp8_max in (0, 448] (448 = e4m3fn max).
 */
int fq_rmsnorm_rope_quant(const void* x, const void* w, const void* cos, const void* sin, void* y,
                          uint8_t* q, float* scale, int64_t M, int64_t N, int64_t rope_dim, int dtype,
                          int table_dtype, float eps, float fp8_max, cudaStream_t stream);

/*
 * RMSNorm + NeoX partial RoPE + FP8 with group-wise scales ("rmsnorm_rope_quant.py",
 * rms_norm_rope_quant_fused, step 3: one fp32 scale per group_size consecutive columns):
 *   y as in fq_rmsnorm_rope (rounded to dtype);
 *   for every row i and group g < G = N / group_size, columns J_g = [g*group_size, (g+1)*group_size):
 *     scale[i*G + g] = max(max_{j in J_g} |y_ij|, 1e-4) / fp8_max               (fp32)
 *     q_ij = e4m3fn_round_to_nearest_even(clamp(y_ij / scale[i*G + g], -fp8_max, fp8_max))
 * y: [M, N] dtype or null; q: [M, N] uint8 e4m3fn codes; scale: [M, G] fp32, row-major.
 * group_size >= 1 must divide N (else FQ_ERR_INVALID_ARG); group_size = N gives exactly
 * fq_rmsnorm_rope_quant. Other arguments and errors as fq_rmsnorm_rope_quant. Group sizes that are
 * multiples of 8 with at most 512 groups per row take the vectorised kernel, others the scalar one.
 */
int fq_rmsnorm_rope_quant_groups(const void* x, const void* w, const void* cos, const void* sin, void* y,
                                 uint8_t* q, float* scale, int64_t M, int64_t N, int64_t rope_dim,
                                 int64_t group_size, int dtype, int table_dtype, float eps, float fp8_max,
                                 cudaStream_t stream);

/*
 * QK-Norm + RoPE + FP8 attention prologue ("case_norm_rope_quant.py", module docstring; design C):
 *   for every token t < T and head h < H = Hq + Hk, the row x = qk[t*token_stride + h*D + (0..D-1)]
 *   is normalised with wq (h < Hq) or wk (h >= Hq), its last R columns are rotated with table row t
 *   (shared by every head of the token), and it is quantised with one fp32 scale per row:
 *     n_j = (x_j * rstd) * w_j;  y = rope(n) as above;  all in fp32 (no rounding to dtype);
 *     scale[t,h] = max(max_j |y_j|, 1e-4) / fp8_max;  q[t,h,j] = e4m3fn(clamp(y_j / scale, +-fp8_max))
 * qk: dtype, token_stride >= H*D elements between consecutive tokens (H*D when packed; larger for
 *     the q/k slice of a fused QKV projection row).
 * wq, wk: [D] dtype. cos, sin: [T, R/2] table_dtype. q_out: [T, H, D] uint8. scale: [T, H] fp32.
 * R = rope_dim: even, 0 <= R <= D. T = 0 is a no-op (pointers may then be null).
 */
int fq_qk_norm_rope_quant(const void* qk, int64_t token_stride, const void* wq, const void* wk,
                          const void* cos, const void* sin, uint8_t* q_out, float* scale, int64_t T,
                          int64_t Hq, int64_t Hk, int64_t D, int64_t rope_dim, int dtype,
                          int table_dtype, float eps, float fp8_max, cudaStream_t stream);

/*
 * The prologue computed as the Ch.28 page's designs ("case_norm_rope_quant.py", default_designs):
 * one CTA per block of rows_per_block consecutive (token, head) rows -- 1 (design A), 8 (design B),
 * Hq + Hk (design C: one whole token) -- each block reading the norm weight and the token's table
 * row through its own L1, so the weight and table are brought from L2 once per block, which is what
 * the page's modelled lookup bytes count. Same results as fq_qk_norm_rope_quant (same arithmetic as
 * its generic kernel). A measurement device, not a fast path. rows_per_block in [1, 128]; needs
 * head_dim = rope_dim <= 128, a multiple of 16, and 16-byte aligned tensors (else
 * FQ_ERR_UNSUPPORTED). Other arguments and errors as fq_qk_norm_rope_quant.
 */
int fq_qk_norm_rope_quant_blocks(const void* qk, int64_t token_stride, const void* wq, const void* wk,
                                 const void* cos, const void* sin, uint8_t* q_out, float* scale, int64_t T,
                                 int64_t Hq, int64_t Hk, int64_t D, int64_t rope_dim, int64_t rows_per_block,
                                 int dtype, int table_dtype, float eps, float fp8_max, cudaStream_t stream);

/*
 * Bytes of caller-provided device workspace fq_rmsnorm_bwd needs for an [M, N] problem: the fp32
 * per-chunk partial column sums of the two-stage dw reduction. 0 when M == 0.
 */
size_t fq_rmsnorm_bwd_workspace_bytes(int64_t M, int64_t N);

/*
 * RMSNorm backward ("rmsnorm_tl.py", RMSNormTileLang.backward), rstd recomputed from x:
 *   xn = x * rstd;  gw = g * w;  c = mean_j(gw_j * xn_j)
 *   dx = dtype(rstd * (gw - xn * c))                  [M, N]
 *   dw = dtype(sum_i g_ij * xn_ij)                    [N]  (fp32 sums)
 * dw is reduced in two deterministic stages: fixed row chunks (a partition that depends only on M)
 * write fp32 partial column sums to `workspace`, then each column sums its chunks in order. The
 * result is bitwise reproducible run to run. dw_f32 (nullable) receives the fp32 sums before the
 * final rounding. workspace: at least fq_rmsnorm_bwd_workspace_bytes(M, N) bytes, 16-byte aligned,
 * no initial contents required. M = 0 writes dw = 0.
 */
int fq_rmsnorm_bwd(const void* x, const void* w, const void* grad_y, void* dx, void* dw, float* dw_f32,
                   void* workspace, size_t workspace_bytes, int64_t M, int64_t N, int dtype, float eps,
                   cudaStream_t stream);

/*
 * RMSNorm backward with the forward's saved rstd ("rmsnorm_tl.py", RMSNormTileLang.backward, with
 * rstd taken from fq_rmsnorm_fwd_rstd instead of recomputed from x): the same dx and dw formulas and
 * the same deterministic two-stage dw, with rstd[i] ([M] fp32, device, not null when M > 0) used for
 * row i; the sum of squares of x is not computed (x is still read for xn = x * rstd). No eps argument:
 * it is inside the saved rstd. Other arguments and errors as fq_rmsnorm_bwd.
 */
int fq_rmsnorm_bwd_rstd(const void* x, const void* w, const void* grad_y, const float* rstd, void* dx, void* dw,
                        float* dw_f32, void* workspace, size_t workspace_bytes, int64_t M, int64_t N, int dtype,
                        cudaStream_t stream);

/* Size of the library's built-in scratch used by fq_rmsnorm_bwd_noalloc (4 MiB of device memory per
 * GPU that loads the library). It fits fq_rmsnorm_bwd_workspace_bytes(M, N) for N <= 4096 at any M,
 * and for wider rows while M is small enough (at most FQ_NOALLOC_SCRATCH_BYTES / (4 * N) chunks). */
#define FQ_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)

/*
 * RMSNorm backward that allocates nothing and takes no workspace. The tutorial pages have no
 * counterpart; it exists for callers that cannot allocate device memory or pass a workspace: for
 * example a plugin inside a framework that owns all device buffers through its own pool and hands
 * the plugin only its tensors, or a latency-critical loop that must never call cudaMalloc (which
 * can synchronise the whole device).
 * Same arguments, results and error rules as fq_rmsnorm_bwd, minus the workspace: the dw partial
 * sums go to a fixed array in the library's own device memory (FQ_NOALLOC_SCRATCH_BYTES per device,
 * held until the process exits). Problems whose fq_rmsnorm_bwd_workspace_bytes(M, N) exceeds that
 * size are rejected with FQ_ERR_INVALID_ARG.
 * The first call on each device looks up that array's device address (with the device current);
 * make that first call before any stream capture. A cudaDeviceReset on that device invalidates the
 * looked-up address: do not call this entry point on that device again in the same process. Every call shares the one array and leaves its
 * contents behind (nothing in it needs clearing: each call overwrites what it reads), so calls
 * that may overlap on the GPU -- on different streams, or from different threads -- race on it and
 * must be serialised by the caller.
 */
int fq_rmsnorm_bwd_noalloc(const void* x, const void* w, const void* grad_y, void* dx, void* dw,
                           float* dw_f32, int64_t M, int64_t N, int dtype, float eps, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FQ_H_ */
