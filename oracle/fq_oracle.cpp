/*
 * fq_oracle.cpp -- reference oracle for the fused RMSNorm -> NeoX partial RoPE -> per-row FP8
 * (e4m3fn) path and for the standalone RMSNorm forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the package smoke check and the benchmark's
 * CPU-baseline leg are the only code that may load this library. The product path (the CUDA
 * library and its Python binding) never calls it, includes nothing from it and shares no code,
 * table or helper with it.
 *
 * Everything here is a plain, single-threaded loop that restates what the tutorial pages define,
 * in their order and at their cast points:
 *
 *   - "rmsnorm_rope_quant.py" (Ch.13 "Operators I: elementwise, normalisation and RoPE", fusion
 *     capstone): `torch_reference_fused` (RMSNorm in fp32, result cast to the storage dtype; NeoX
 *     rotation of the last rope_dim columns in fp32, cast back; row amax clamped at 1e-4,
 *     scale = amax / fp8_max, q = e4m3fn(y / scale)) and `_torch_rope_neox` (pairs (p, p+half)).
 *     The kernel `rms_norm_rope_quant_fused` adds the clamp to +-fp8_max before the cast.
 *   - "rmsnorm_tl.py" (Ch.17 "End to end I: training a 7B model"): `_rmsnorm_fwd` (fp32
 *     accumulation, one rounding of x*rstd*w) and `RMSNormTileLang.backward`
 *     (rstd recomputed; xn = x*rstd; dw = sum over rows of g*xn; dx = rstd*(g*w - xn*mean(g*w*xn))).
 *   - "case_norm_rope_quant.py" (Ch.28 "Operator design methodology", module docstring): the
 *     QK-Norm + RoPE + FP8 prologue over [tokens, heads, head_dim], RMSNorm per (token, head),
 *     one cos/sin row per token shared by every head, one fp32 scale per row.
 *
 * Readings taken where the pages leave a step open (each one is listed in the design notes):
 *   - Sum of squares: the exact sum of the (exact) squares, accumulated in fp64 and rounded once
 *     to fp32. The pages name an fp32 reduction without an order.
 *   - rsqrt(v) is 1/sqrt(v) with both the square root and the division correctly rounded in fp32.
 *   - The prologue has no y output, so it keeps fp32 from the load to the quantiser (no rounding of
 *     the normalised or rotated row to the storage dtype). rmsnorm_rope / rmsnorm_rope_quant keep
 *     the fusion page's two roundings to the storage dtype.
 *   - cos/sin tables are inputs (built by the input generator), half width [rows, rope_dim/2].
 *   - Quantisation divides (true fp32 division), clamps to +-fp8_max, then rounds to nearest even.
 *   - dw is the fp64-accumulated column sum of the fp32 products g*xn, rounded once to fp32 and
 *     then to the storage dtype.
 *
 *   - LayerNorm ("ledger.py", Ch.13 ledger, layer_norm: y = (x - mean) / sqrt(var + eps) * g + b, one
 *     fused kernel reading x, g, b and writing y): the page gives the formula only; this follows the
 *     RMSNorm conventions above -- the row's mean and variance (mean of (x - mean)^2) from exact
 *     fp64 sums rounded once to fp32, rstd = 1/sqrt(var + eps) in fp32, then
 *     y = dtype(((x - mean) * rstd) * g + b) with every fp32 step rounded.
 *
 * Build: g++ -O2 -std=c++17 -ffp-contract=off -fno-fast-math -fPIC -shared (oracle/build.py).
 * -ffp-contract=off matters: every a*b+c below is two roundings, as in the fp32 tensor ops of the
 * pages' reference code.
 */
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ------------------------------------------------------------------------------------------------
// Storage formats, written from the format definitions.
//   bf16:    1 sign, 8 exponent (bias 127), 7 fraction bits; IEEE-style inf/NaN.
//   fp16:    IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
//   e4m3fn:  OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 fraction bits; no infinities; the only
//            NaN encodings are S.1111.111; largest finite magnitude 1.110b x 2^8 = 448.
// Rounding is to nearest, ties to even, at the format's precision (subnormals included).
// ------------------------------------------------------------------------------------------------
enum Fmt { FMT_BF16 = 0, FMT_F16 = 1, FMT_F32 = 2, FMT_E4M3 = 3 };

struct Layout {
  int ebits, mbits, bias;
  bool ieee_specials;  // all-ones exponent field = inf/NaN (bf16, fp16); false for e4m3fn
};

Layout layout_of(int fmt) {
  switch (fmt) {
    case FMT_BF16: return {8, 7, 127, true};
    case FMT_F16: return {5, 10, 15, true};
    default: return {4, 3, 7, false};  // FMT_E4M3
  }
}

uint32_t encode_binary(double v, const Layout& L) {
  const uint32_t sign = std::signbit(v) ? 1u : 0u;
  const uint32_t sign_bit = sign << (L.ebits + L.mbits);
  const uint32_t exp_all_ones = (1u << L.ebits) - 1u;
  if (std::isnan(v)) {
    if (L.ieee_specials) return sign_bit | (exp_all_ones << L.mbits) | (1u << (L.mbits - 1));
    return sign_bit | (exp_all_ones << L.mbits) | ((1u << L.mbits) - 1u);
  }
  double a = std::fabs(v);
  if (std::isinf(a)) {
    if (L.ieee_specials) return sign_bit | (exp_all_ones << L.mbits);
    return sign_bit | (exp_all_ones << L.mbits) | ((1u << L.mbits) - 1u);  // e4m3fn: NaN
  }
  if (a == 0.0) return sign_bit;
  const int emin = 1 - L.bias;  // exponent of the smallest normal number
  int e2 = 0;
  std::frexp(a, &e2);  // a = f * 2^e2 with f in [0.5, 1)
  int E = e2 - 1;      // a = 1.fff * 2^E
  if (E < emin) E = emin;  // subnormal range: same quantum as the smallest binade
  // Quantum (one unit in the last place) at exponent E; a / quantum is exact (power of two).
  const double scaled = std::ldexp(a, L.mbits - E);
  double n = std::nearbyint(scaled);  // current mode is round-to-nearest-even
  const double hidden = std::ldexp(1.0, L.mbits);
  if (n >= 2.0 * hidden) {  // rounded up into the next binade
    n = hidden;
    E += 1;
  }
  uint32_t exp_field, mant;
  if (n < hidden) {  // subnormal (only reachable with E == emin)
    exp_field = 0;
    mant = static_cast<uint32_t>(n);
  } else {
    exp_field = static_cast<uint32_t>(E + L.bias);
    mant = static_cast<uint32_t>(n - hidden);
  }
  if (L.ieee_specials) {
    if (exp_field >= exp_all_ones) return sign_bit | (exp_all_ones << L.mbits);  // overflow: inf
  } else {
    // e4m3fn: exponent field 15 with fraction 111 is NaN; anything larger overflows to NaN.
    if (exp_field > exp_all_ones || (exp_field == exp_all_ones && mant == (1u << L.mbits) - 1u))
      return sign_bit | (exp_all_ones << L.mbits) | ((1u << L.mbits) - 1u);
  }
  return sign_bit | (exp_field << L.mbits) | mant;
}

double decode_binary(uint32_t code, const Layout& L) {
  const uint32_t mant = code & ((1u << L.mbits) - 1u);
  const uint32_t exp_field = (code >> L.mbits) & ((1u << L.ebits) - 1u);
  const bool neg = (code >> (L.ebits + L.mbits)) & 1u;
  const uint32_t exp_all_ones = (1u << L.ebits) - 1u;
  double mag;
  if (L.ieee_specials && exp_field == exp_all_ones) {
    mag = mant ? NAN : INFINITY;
  } else if (!L.ieee_specials && exp_field == exp_all_ones && mant == (1u << L.mbits) - 1u) {
    mag = NAN;
  } else if (exp_field == 0) {
    mag = std::ldexp(static_cast<double>(mant), 1 - L.bias - L.mbits);
  } else {
    mag = std::ldexp(static_cast<double>((1u << L.mbits) + mant),
                     static_cast<int>(exp_field) - L.bias - L.mbits);
  }
  return neg ? -mag : mag;
}

// Value of element i of a stored array in format fmt (bf16 / fp16 stored as 16-bit patterns).
float load_elem(int fmt, const void* p, int64_t i) {
  if (fmt == FMT_F32) return static_cast<const float*>(p)[i];
  const uint16_t bits = static_cast<const uint16_t*>(p)[i];
  return static_cast<float>(decode_binary(bits, layout_of(fmt)));
}

void store_elem(int fmt, void* p, int64_t i, float v) {
  if (fmt == FMT_F32) {
    static_cast<float*>(p)[i] = v;
    return;
  }
  static_cast<uint16_t*>(p)[i] = static_cast<uint16_t>(encode_binary(v, layout_of(fmt)));
}

// v rounded to the storage format (the `.to(x.dtype)` cast of the pages' reference code).
float round_to(int fmt, float v) {
  if (fmt == FMT_F32) return v;
  return static_cast<float>(decode_binary(encode_binary(v, layout_of(fmt)), layout_of(fmt)));
}

uint8_t e4m3_encode(float v) { return static_cast<uint8_t>(encode_binary(v, layout_of(FMT_E4M3))); }

bool is_storage(int fmt) { return fmt == FMT_BF16 || fmt == FMT_F16; }
bool is_table(int fmt) { return fmt == FMT_BF16 || fmt == FMT_F16 || fmt == FMT_F32; }

// ------------------------------------------------------------------------------------------------
// Step a2: rstd of one row.  Sum of squares accumulated in fp64 (each square of a bf16/fp16 value
// is exact), rounded once to fp32; then mean = ss / N, + eps and 1/sqrt in fp32.
// ------------------------------------------------------------------------------------------------
float row_rstd(const float* xr, int64_t N, float eps) {
  double ss = 0.0;
  for (int64_t j = 0; j < N; ++j) ss += static_cast<double>(xr[j]) * static_cast<double>(xr[j]);
  const float ss32 = static_cast<float>(ss);
  const float mean = ss32 / static_cast<float>(N);
  const float v = mean + eps;
  return 1.0f / std::sqrt(v);
}

// Step a4: NeoX rotation of the last R columns of one fp32 row, in place, in fp32.
// For p < R/2: lo = row[N-R+p], hi = row[N-R+R/2+p];
//   lo' = lo*c - hi*s,  hi' = hi*c + lo*s   (each product rounded, then the sum).
void rope_tail_f32(float* row, int64_t N, int64_t R, const float* c, const float* s) {
  const int64_t half = R / 2;
  const int64_t base = N - R;
  for (int64_t p = 0; p < half; ++p) {
    const float lo = row[base + p];
    const float hi = row[base + half + p];
    const float lo_c = lo * c[p];
    const float hi_s = hi * s[p];
    const float hi_c = hi * c[p];
    const float lo_s = lo * s[p];
    row[base + p] = lo_c - hi_s;
    row[base + half + p] = hi_c + lo_s;
  }
}

// Steps a6-a7 on one fp32 row y: amax, scale and codes.
float quant_row(const float* y, int64_t N, float fp8_max, uint8_t* q) {
  float amax = 0.0f;
  for (int64_t j = 0; j < N; ++j) amax = std::fmax(amax, std::fabs(y[j]));
  amax = std::fmax(amax, 1e-4f);  // clamp(min=1e-4)
  const float scale = amax / fp8_max;
  for (int64_t j = 0; j < N; ++j) {
    float v = y[j] / scale;
    if (v > fp8_max) v = fp8_max;
    if (v < -fp8_max) v = -fp8_max;
    q[j] = e4m3_encode(v);
  }
  return scale;
}

// Step 3 of "rms_norm_rope_quant_fused" on one fp32 row: the row viewed as n_groups = N / gs groups
// of gs consecutive columns; per group, amax of |y| clamped at 1e-4, scale = amax / fp8_max, and
// every element of the group divided by its group's scale, clamped to +-fp8_max, rounded to e4m3fn.
void quant_groups(const float* y, int64_t N, int64_t gs, float fp8_max, uint8_t* q, float* scale) {
  const int64_t n_groups = N / gs;
  for (int64_t g = 0; g < n_groups; ++g) {
    const float* yg = y + g * gs;
    float amax = 0.0f;
    for (int64_t k = 0; k < gs; ++k) amax = std::fmax(amax, std::fabs(yg[k]));
    const float sc = std::fmax(amax, 1e-4f) / fp8_max;
    for (int64_t k = 0; k < gs; ++k) {
      float v = yg[k] / sc;
      if (v > fp8_max) v = fp8_max;
      if (v < -fp8_max) v = -fp8_max;
      q[g * gs + k] = e4m3_encode(v);
    }
    scale[g] = sc;
  }
}

}  // namespace

extern "C" {

// Status codes of the oracle entry points.
enum { OR_OK = 0, OR_BAD_ARG = 1 };

// ---- format conversion (for the format pins) ----
// fmt: 0 bf16, 1 fp16, 2 fp32 (copy), 3 e4m3fn. 16-bit formats are uint16 patterns, e4m3 uint8.
int or_encode(int fmt, const float* src, void* dst, int64_t n) {
  if (!src || !dst || n < 0 || fmt < 0 || fmt > 3) return OR_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (fmt == FMT_F32) static_cast<float*>(dst)[i] = src[i];
    else if (fmt == FMT_E4M3) static_cast<uint8_t*>(dst)[i] = e4m3_encode(src[i]);
    else static_cast<uint16_t*>(dst)[i] = static_cast<uint16_t>(encode_binary(src[i], layout_of(fmt)));
  }
  return OR_OK;
}

int or_decode(int fmt, const void* src, float* dst, int64_t n) {
  if (!src || !dst || n < 0 || fmt < 0 || fmt > 3) return OR_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (fmt == FMT_F32) dst[i] = static_cast<const float*>(src)[i];
    else if (fmt == FMT_E4M3)
      dst[i] = static_cast<float>(decode_binary(static_cast<const uint8_t*>(src)[i], layout_of(FMT_E4M3)));
    else dst[i] = static_cast<float>(decode_binary(static_cast<const uint16_t*>(src)[i], layout_of(fmt)));
  }
  return OR_OK;
}

// ---- b1: RMSNorm forward, y = dtype(x * rstd * w), one rounding ("rmsnorm_tl.py", _rmsnorm_fwd)
int or_rmsnorm_fwd(const void* x, const void* w, void* y, int64_t M, int64_t N, int dtype, float eps) {
  if (!x || !w || !y || M < 0 || N <= 0 || !is_storage(dtype)) return OR_BAD_ARG;
  std::vector<float> xr(N), wr(N);
  for (int64_t j = 0; j < N; ++j) wr[j] = load_elem(dtype, w, j);
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) xr[j] = load_elem(dtype, x, i * N + j);
    const float rstd = row_rstd(xr.data(), N, eps);
    for (int64_t j = 0; j < N; ++j) store_elem(dtype, y, i * N + j, (xr[j] * rstd) * wr[j]);
  }
  return OR_OK;
}

// Shared row body of rmsnorm_rope / rmsnorm_rope_quant ("rmsnorm_rope_quant.py",
// torch_reference_fused): normed = dtype(x*rstd*w); y = cat(head, dtype(rope(tail))).
static void normed_rope_row(int dtype, int tdtype, const void* x, const float* wr, const void* cs,
                            const void* sn, int64_t i, int64_t N, int64_t R, float eps, float* xr,
                            float* yr, float* cr, float* sr) {
  for (int64_t j = 0; j < N; ++j) xr[j] = load_elem(dtype, x, i * N + j);
  const float rstd = row_rstd(xr, N, eps);
  for (int64_t j = 0; j < N; ++j) yr[j] = round_to(dtype, (xr[j] * rstd) * wr[j]);
  const int64_t half = R / 2;
  for (int64_t p = 0; p < half; ++p) {
    cr[p] = load_elem(tdtype, cs, i * half + p);
    sr[p] = load_elem(tdtype, sn, i * half + p);
  }
  rope_tail_f32(yr, N, R, cr, sr);
  for (int64_t j = N - R; j < N; ++j) yr[j] = round_to(dtype, yr[j]);
}

// ---- a1-a5: RMSNorm + NeoX partial RoPE, y written in dtype ("rmsnorm_rope_quant.py",
// torch_reference_fused without the quantiser; kernel rms_norm_rope_fused)
int or_rmsnorm_rope(const void* x, const void* w, const void* cs, const void* sn, void* y, int64_t M,
                    int64_t N, int64_t R, int dtype, int tdtype, float eps) {
  if (!x || !w || (R > 0 && (!cs || !sn)) || !y || M < 0 || N <= 0 || R < 0 || R % 2 || R > N ||
      !is_storage(dtype) || !is_table(tdtype))
    return OR_BAD_ARG;
  std::vector<float> wr(N), xr(N), yr(N), cr(R / 2 + 1), sr(R / 2 + 1);
  for (int64_t j = 0; j < N; ++j) wr[j] = load_elem(dtype, w, j);
  for (int64_t i = 0; i < M; ++i) {
    normed_rope_row(dtype, tdtype, x, wr.data(), cs, sn, i, N, R, eps, xr.data(), yr.data(), cr.data(),
                    sr.data());
    for (int64_t j = 0; j < N; ++j) store_elem(dtype, y, i * N + j, yr[j]);
  }
  return OR_OK;
}

// ---- a1-a8: RMSNorm + RoPE + per-row FP8 ("rmsnorm_rope_quant.py", torch_reference_fused).
// y may be null (not written); q and scale are always written.
int or_rmsnorm_rope_quant(const void* x, const void* w, const void* cs, const void* sn, void* y,
                          uint8_t* q, float* scale, int64_t M, int64_t N, int64_t R, int dtype,
                          int tdtype, float eps, float fp8_max) {
  if (!x || !w || (R > 0 && (!cs || !sn)) || !q || !scale || M < 0 || N <= 0 || R < 0 || R % 2 || R > N ||
      !is_storage(dtype) || !is_table(tdtype) || !(fp8_max > 0.0f) || fp8_max > 448.0f)
    return OR_BAD_ARG;
  std::vector<float> wr(N), xr(N), yr(N), cr(R / 2 + 1), sr(R / 2 + 1);
  for (int64_t j = 0; j < N; ++j) wr[j] = load_elem(dtype, w, j);
  for (int64_t i = 0; i < M; ++i) {
    normed_rope_row(dtype, tdtype, x, wr.data(), cs, sn, i, N, R, eps, xr.data(), yr.data(), cr.data(),
                    sr.data());
    if (y)
      for (int64_t j = 0; j < N; ++j) store_elem(dtype, y, i * N + j, yr[j]);
    scale[i] = quant_row(yr.data(), N, fp8_max, q + i * N);
  }
  return OR_OK;
}

// ---- a6-a8 alone on a stored y (lets a test check a fused kernel's codes against its own y).
int or_quant_rows(const void* y, uint8_t* q, float* scale, int64_t M, int64_t N, int dtype,
                  float fp8_max) {
  if (!y || !q || !scale || M < 0 || N <= 0 || !is_table(dtype) || !(fp8_max > 0.0f) ||
      fp8_max > 448.0f)
    return OR_BAD_ARG;
  std::vector<float> yr(N);
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) yr[j] = load_elem(dtype, y, i * N + j);
    scale[i] = quant_row(yr.data(), N, fp8_max, q + i * N);
  }
  return OR_OK;
}

// ---- a1-a8 with group-wise scales ("rmsnorm_rope_quant.py", rms_norm_rope_quant_fused: one fp32
// scale per group_size consecutive columns, Scale[M, N / group_size]). N % group_size == 0.
int or_rmsnorm_rope_quant_groups(const void* x, const void* w, const void* cs, const void* sn, void* y,
                                 uint8_t* q, float* scale, int64_t M, int64_t N, int64_t R, int64_t gs,
                                 int dtype, int tdtype, float eps, float fp8_max) {
  if (!x || !w || (R > 0 && (!cs || !sn)) || !q || !scale || M < 0 || N <= 0 || R < 0 || R % 2 || R > N ||
      gs < 1 || N % gs != 0 || !is_storage(dtype) || !is_table(tdtype) || !(fp8_max > 0.0f) ||
      fp8_max > 448.0f)
    return OR_BAD_ARG;
  const int64_t n_groups = N / gs;
  std::vector<float> wr(N), xr(N), yr(N), cr(R / 2 + 1), sr(R / 2 + 1);
  for (int64_t j = 0; j < N; ++j) wr[j] = load_elem(dtype, w, j);
  for (int64_t i = 0; i < M; ++i) {
    normed_rope_row(dtype, tdtype, x, wr.data(), cs, sn, i, N, R, eps, xr.data(), yr.data(), cr.data(),
                    sr.data());
    if (y)
      for (int64_t j = 0; j < N; ++j) store_elem(dtype, y, i * N + j, yr[j]);
    quant_groups(yr.data(), N, gs, fp8_max, q + i * N, scale + i * n_groups);
  }
  return OR_OK;
}

// ---- the group-wise quantiser alone on a stored y
int or_quant_groups(const void* y, uint8_t* q, float* scale, int64_t M, int64_t N, int64_t gs, int dtype,
                    float fp8_max) {
  if (!y || !q || !scale || M < 0 || N <= 0 || gs < 1 || N % gs != 0 || !is_table(dtype) ||
      !(fp8_max > 0.0f) || fp8_max > 448.0f)
    return OR_BAD_ARG;
  std::vector<float> yr(N);
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) yr[j] = load_elem(dtype, y, i * N + j);
    quant_groups(yr.data(), N, gs, fp8_max, q + i * N, scale + i * (N / gs));
  }
  return OR_OK;
}

// ---- LayerNorm forward ("ledger.py", Ch.13 ledger, layer_norm). b may be null (no bias). Also writes
// each row's fp32 mean and rstd when those pointers are given.
int or_layernorm_fwd(const void* x, const void* g, const void* b, void* y, float* mean_out, float* rstd_out,
                     int64_t M, int64_t N, int dtype, float eps) {
  if (!x || !g || !y || M < 0 || N <= 0 || !is_storage(dtype)) return OR_BAD_ARG;
  std::vector<float> xr(N), gr(N), br(N, 0.0f);
  for (int64_t j = 0; j < N; ++j) {
    gr[j] = load_elem(dtype, g, j);
    if (b) br[j] = load_elem(dtype, b, j);
  }
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) xr[j] = load_elem(dtype, x, i * N + j);
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j) s += static_cast<double>(xr[j]);
    const double mean64 = s / static_cast<double>(N);
    double v = 0.0;
    for (int64_t j = 0; j < N; ++j) v += (static_cast<double>(xr[j]) - mean64) * (static_cast<double>(xr[j]) - mean64);
    const float mean = static_cast<float>(mean64);
    const float var = static_cast<float>(v / static_cast<double>(N));
    const float rstd = 1.0f / std::sqrt(var + eps);
    if (mean_out) mean_out[i] = mean;
    if (rstd_out) rstd_out[i] = rstd;
    for (int64_t j = 0; j < N; ++j) {
      const float c = xr[j] - mean;
      store_elem(dtype, y, i * N + j, ((c * rstd) * gr[j]) + br[j]);
    }
  }
  return OR_OK;
}

// ---- The QK-Norm + RoPE + FP8 prologue ("case_norm_rope_quant.py", module docstring).
// qk: [T, token_stride] storage elements; row (t, h) starts at t*token_stride + h*D, h < Hq+Hk.
// Heads [0, Hq) use wq, heads [Hq, Hq+Hk) use wk. cos/sin: [T, R/2], one row per token.
// q: [T, Hq+Hk, D] e4m3fn codes; scale: [T, Hq+Hk] fp32.  fp32 from load to quantiser.
int or_qk_norm_rope_quant(const void* qk, int64_t token_stride, const void* wq, const void* wk,
                          const void* cs, const void* sn, uint8_t* q, float* scale, int64_t T,
                          int64_t Hq, int64_t Hk, int64_t D, int64_t R, int dtype, int tdtype,
                          float eps, float fp8_max) {
  const int64_t H = Hq + Hk;
  if (!qk || !wq || !wk || (R > 0 && (!cs || !sn)) || !q || !scale || T < 0 || Hq < 0 || Hk < 0 || H <= 0 ||
      D <= 0 || R < 0 || R % 2 || R > D || token_stride < H * D || !is_storage(dtype) ||
      !is_table(tdtype) || !(fp8_max > 0.0f) || fp8_max > 448.0f)
    return OR_BAD_ARG;
  std::vector<float> wqr(D), wkr(D), xr(D), yr(D), cr(R / 2 + 1), sr(R / 2 + 1);
  for (int64_t j = 0; j < D; ++j) {
    wqr[j] = load_elem(dtype, wq, j);
    wkr[j] = load_elem(dtype, wk, j);
  }
  const int64_t half = R / 2;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t p = 0; p < half; ++p) {
      cr[p] = load_elem(tdtype, cs, t * half + p);
      sr[p] = load_elem(tdtype, sn, t * half + p);
    }
    for (int64_t h = 0; h < H; ++h) {
      const float* wr = (h < Hq) ? wqr.data() : wkr.data();
      for (int64_t j = 0; j < D; ++j) xr[j] = load_elem(dtype, qk, t * token_stride + h * D + j);
      const float rstd = row_rstd(xr.data(), D, eps);
      for (int64_t j = 0; j < D; ++j) yr[j] = (xr[j] * rstd) * wr[j];
      rope_tail_f32(yr.data(), D, R, cr.data(), sr.data());
      const int64_t r = t * H + h;
      scale[r] = quant_row(yr.data(), D, fp8_max, q + r * D);
    }
  }
  return OR_OK;
}

// ---- b2-b3: RMSNorm backward ("rmsnorm_tl.py", RMSNormTileLang.backward).
// dx = dtype(rstd*(g*w - xn*mean(g*w*xn))), dw = dtype(sum_rows g*xn). dw_f32 (nullable) receives
// the fp32 column sums before the final cast.
// Shared body of the backward: rstd recomputed from x (as the Ch.17 page does) or, when `rstd_in` is
// given, the forward's saved rstd of each row.
static int bwd_impl(const void* x, const void* w, const void* g, const float* rstd_in, void* dx, void* dw,
                    float* dw_f32, int64_t M, int64_t N, int dtype, float eps) {
  if (!x || !w || !g || !dx || !dw || M < 0 || N <= 0 || !is_storage(dtype)) return OR_BAD_ARG;
  std::vector<float> wr(N), xr(N), xn(N), gw(N);
  std::vector<double> dw_acc(N, 0.0);
  for (int64_t j = 0; j < N; ++j) wr[j] = load_elem(dtype, w, j);
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) xr[j] = load_elem(dtype, x, i * N + j);
    const float rstd = rstd_in ? rstd_in[i] : row_rstd(xr.data(), N, eps);
    double tsum = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      const float gj = load_elem(dtype, g, i * N + j);
      xn[j] = xr[j] * rstd;
      dw_acc[j] += static_cast<double>(gj * xn[j]);
      gw[j] = gj * wr[j];
      tsum += static_cast<double>(gw[j] * xn[j]);
    }
    const float c = static_cast<float>(tsum) / static_cast<float>(N);  // mean(g*w*xn)
    for (int64_t j = 0; j < N; ++j) {
      const float xc = xn[j] * c;
      const float d = gw[j] - xc;
      store_elem(dtype, dx, i * N + j, rstd * d);
    }
  }
  for (int64_t j = 0; j < N; ++j) {
    const float s = static_cast<float>(dw_acc[j]);
    if (dw_f32) dw_f32[j] = s;
    store_elem(dtype, dw, j, s);
  }
  return OR_OK;
}

int or_rmsnorm_bwd(const void* x, const void* w, const void* g, void* dx, void* dw, float* dw_f32,
                   int64_t M, int64_t N, int dtype, float eps) {
  return bwd_impl(x, w, g, nullptr, dx, dw, dw_f32, M, N, dtype, eps);
}

// ---- b2-b3 with the forward's rstd saved instead of recomputed (a trade of a 4-byte-per-row write
// and read for the backward's sum of squares).
int or_rmsnorm_bwd_rstd(const void* x, const void* w, const void* g, const float* rstd, void* dx, void* dw,
                        float* dw_f32, int64_t M, int64_t N, int dtype) {
  if (!rstd && M > 0) return OR_BAD_ARG;
  return bwd_impl(x, w, g, rstd, dx, dw, dw_f32, M, N, dtype, 0.0f);
}

// ---- b1 that also returns each row's rstd = 1/sqrt(mean(x^2) + eps) (fp32), for the backward.
int or_rmsnorm_fwd_rstd(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N, int dtype,
                        float eps) {
  if (!x || !w || !y || !rstd || M < 0 || N <= 0 || !is_storage(dtype)) return OR_BAD_ARG;
  std::vector<float> xr(N), wr(N);
  for (int64_t j = 0; j < N; ++j) wr[j] = load_elem(dtype, w, j);
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) xr[j] = load_elem(dtype, x, i * N + j);
    rstd[i] = row_rstd(xr.data(), N, eps);
    for (int64_t j = 0; j < N; ++j) store_elem(dtype, y, i * N + j, (xr[j] * rstd[i]) * wr[j]);
  }
  return OR_OK;
}

// ---- fp64 twins of the same definitions: used only to pin the fp32 oracle (invariants that are
// exact in real arithmetic, central finite differences for the backward).
int or_layernorm_f64(const double* x, const double* g, const double* b, double* y, int64_t M, int64_t N,
                     double eps) {
  if (!x || !g || !y || M < 0 || N <= 0) return OR_BAD_ARG;
  for (int64_t i = 0; i < M; ++i) {
    const double* xr = x + i * N;
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j) s += xr[j];
    const double mean = s / static_cast<double>(N);
    double v = 0.0;
    for (int64_t j = 0; j < N; ++j) v += (xr[j] - mean) * (xr[j] - mean);
    const double rstd = 1.0 / std::sqrt(v / static_cast<double>(N) + eps);
    for (int64_t j = 0; j < N; ++j) y[i * N + j] = (xr[j] - mean) * rstd * g[j] + (b ? b[j] : 0.0);
  }
  return OR_OK;
}

int or_rmsnorm_f64(const double* x, const double* w, double* y, int64_t M, int64_t N, double eps) {
  if (!x || !w || !y || M < 0 || N <= 0) return OR_BAD_ARG;
  for (int64_t i = 0; i < M; ++i) {
    double ss = 0.0;
    for (int64_t j = 0; j < N; ++j) ss += x[i * N + j] * x[i * N + j];
    const double rstd = 1.0 / std::sqrt(ss / static_cast<double>(N) + eps);
    for (int64_t j = 0; j < N; ++j) y[i * N + j] = x[i * N + j] * rstd * w[j];
  }
  return OR_OK;
}

int or_rope_f64(double* rows, const double* cs, const double* sn, int64_t M, int64_t N, int64_t R) {
  if (!rows || (R > 0 && (!cs || !sn)) || M < 0 || N <= 0 || R < 0 || R % 2 || R > N) return OR_BAD_ARG;
  const int64_t half = R / 2;
  for (int64_t i = 0; i < M; ++i) {
    double* row = rows + i * N;
    for (int64_t p = 0; p < half; ++p) {
      const double lo = row[N - R + p], hi = row[N - R + half + p];
      const double c = cs[i * half + p], s = sn[i * half + p];
      row[N - R + p] = lo * c - hi * s;
      row[N - R + half + p] = hi * c + lo * s;
    }
  }
  return OR_OK;
}

int or_rmsnorm_bwd_f64(const double* x, const double* w, const double* g, double* dx, double* dw,
                       int64_t M, int64_t N, double eps) {
  if (!x || !w || !g || !dx || !dw || M < 0 || N <= 0) return OR_BAD_ARG;
  for (int64_t j = 0; j < N; ++j) dw[j] = 0.0;
  std::vector<double> xn(N), gw(N);
  for (int64_t i = 0; i < M; ++i) {
    double ss = 0.0;
    for (int64_t j = 0; j < N; ++j) ss += x[i * N + j] * x[i * N + j];
    const double rstd = 1.0 / std::sqrt(ss / static_cast<double>(N) + eps);
    double tsum = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      xn[j] = x[i * N + j] * rstd;
      gw[j] = g[i * N + j] * w[j];
      dw[j] += g[i * N + j] * xn[j];
      tsum += gw[j] * xn[j];
    }
    const double c = tsum / static_cast<double>(N);
    for (int64_t j = 0; j < N; ++j) dx[i * N + j] = rstd * (gw[j] - xn[j] * c);
  }
  return OR_OK;
}

}  // extern "C"
