/*
 * RMSNorm oracle: plain, slow, double-precision CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * bench's CPU-baseline / reference arm may load or run this file; the CUDA
 * library never links it and shares no code with it.
 *
 * What it computes (definitions from "Pre-built kernel library guide" (FlyDSL),
 * section 1.2 RMSNorm):
 *   forward      RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma, per row of an
 *                M x N row-major matrix; rstd = 1 / sqrt(mean(x^2) + eps) is the
 *                optional per-row output that the backward reads, so eps is
 *                folded into rstd and the backward does not need it.
 *   fused add    the residual-add variant named in "TIRx kernels", Kernels list
 *                (flashinfer.norm: fused_add_rmsnorm): h = residual + x, stored in
 *                the activation dtype, then y = RMSNorm(h) * gamma of that stored h.
 *   backward     dx and the weight gradient of the forward (same section: reads
 *                Input, Gamma, DY, Rstd; writes DX and DWeight).  The pages give
 *                no formula; differentiating y_j = gamma_j x_j r with
 *                r = (sum_k x_k^2 / N + eps)^(-1/2) gives
 *                  dx_j     = r (gamma_j dy_j - x_j c),  c = r^2/N sum_k gamma_k dy_k x_k
 *                  dgamma_j = sum_rows dy_j x_j r
 *                with r the saved rstd when one is given.
 *   layernorm    (x - mean) / sqrt(var + eps) * gamma + beta (same guide,
 *                section 1.1), two passes (mean, then the population variance
 *                about it), and its backward, derived below.
 *   quantised    the forward (and the fused add) with an FP8 E4M3 output and
 *                one scale per row, or an NVFP4 output (FP4 E2M1 codes with an
 *                E4M3 scale per 16 elements and a global scale); the pages name
 *                these ops only, the formulas below each function are the
 *                plain readings of those names.
 *
 * Every sum is a plain left-to-right double-precision loop; every stored
 * output is rounded once, from double, to its dtype (round to nearest even).
 * Pins: all functions are pinned by the CPU tests (closed forms, the eps = 0
 * invariants, the backward orthogonality identity, central finite differences,
 * library routines on special cases, hand-derived fixtures).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* ---- storage types -------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32: widen the bits, reinterpret. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t w = (uint32_t)b << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* Nearest bf16 to v, ties to even, straight from double (no fp32 step, which
 * could round twice).  bf16: sign, 8-bit exponent (bias 127), 7-bit fraction;
 * subnormals below 2^-126 with spacing 2^-133; overflow to infinity. */
uint16_t oracle_round_bf16(double v) {
  if (v != v) return 0x7FC0;                       /* NaN stays NaN */
  uint16_t s = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (isinf(a)) return (uint16_t)(s | 0x7F80u);
  /* find the binade: 2^k <= a < 2^(k+1); spacing of bf16 there is 2^(k-7) */
  int k;
  if (a == 0.0) return s;
  frexp(a, &k);
  k -= 1;
  if (k < -126) k = -126;
  double ulp = ldexp(1.0, k - 7);
  double n = a / ulp;                              /* exact (power of two) */
  double lo = floor(n);
  double frac = n - lo;
  double m = lo;
  if (frac > 0.5) m = lo + 1.0;
  else if (frac == 0.5) m = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
  /* m * ulp is the rounded magnitude; m in [0, 256] */
  double rounded = m * ulp;
  if (rounded > 3.3895313892515355e38) return (uint16_t)(s | 0x7F80u); /* > max finite */
  float rf = (float)rounded;                       /* exact: 8 significant bits */
  uint32_t w;
  memcpy(&w, &rf, sizeof w);
  return (uint16_t)(s | (uint16_t)((w >> 16) & 0x7FFFu));
}

static double load(const void* p, int dt, int64_t i) {
  if (dt == ORACLE_F32) return (double)((const float*)p)[i];
  return oracle_bf16_to_double(((const uint16_t*)p)[i]);
}

static void store(void* p, int dt, int64_t i, double v) {
  if (dt == ORACLE_F32)
    ((float*)p)[i] = (float)v;                     /* C conversion: nearest even */
  else
    ((uint16_t*)p)[i] = oracle_round_bf16(v);
}

static int bad_dtypes(int x_dtype, int w_dtype) {
  if (x_dtype == ORACLE_F32) return w_dtype != ORACLE_F32;
  if (x_dtype == ORACLE_BF16) return w_dtype != ORACLE_F32 && w_dtype != ORACLE_BF16;
  return 1;
}

/* ---- forward ------------------------------------------------------------- */

/* One row: r = 1/sqrt(mean(v^2) + eps), y = v * r * gamma. */
static void fwd_row(const double* v, const void* gamma, int w_dtype, int64_t N, double eps,
                    double* r_out, double* y_row) {
  double ss = 0.0;
  for (int64_t j = 0; j < N; ++j) ss += v[j] * v[j];
  double mean_sq = ss / (double)N;
  double r = 1.0 / sqrt(mean_sq + eps);
  *r_out = r;
  for (int64_t j = 0; j < N; ++j) y_row[j] = v[j] * r * load(gamma, w_dtype, j);
}

/* x: M x N (x_dtype); gamma: N (w_dtype).  Outputs (each may be NULL):
 * y (x_dtype, rounded once), y64 (exact-ish double), rstd (fp32, rounded once),
 * rstd64 (double).  Returns 0, or -1 on bad arguments. */
int oracle_rmsnorm_fwd(const void* x, const void* gamma, int64_t M, int64_t N, double eps,
                       int x_dtype, int w_dtype, void* y, double* y64, float* rstd,
                       double* rstd64) {
  if (M < 0 || N <= 0 || bad_dtypes(x_dtype, w_dtype) || (M > 0 && (!x || !gamma)))
    return -1;
  double* v = (double*)malloc((size_t)N * sizeof(double));
  double* yr = (double*)malloc((size_t)N * sizeof(double));
  if (!v || !yr) { free(v); free(yr); return -1; }
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) v[j] = load(x, x_dtype, i * N + j);
    double r;
    fwd_row(v, gamma, w_dtype, N, eps, &r, yr);
    if (rstd) rstd[i] = (float)r;
    if (rstd64) rstd64[i] = r;
    for (int64_t j = 0; j < N; ++j) {
      if (y) store(y, x_dtype, i * N + j, yr[j]);
      if (y64) y64[i * N + j] = yr[j];
    }
  }
  free(v);
  free(yr);
  return 0;
}

/* ---- fused residual add + forward ---------------------------------------- */

/* h = residual + x rounded to x_dtype (the stored new residual), then the
 * forward of that stored h.  residual is read only; h is a separate output
 * (may be NULL).  Other outputs as in oracle_rmsnorm_fwd. */
int oracle_rmsnorm_fused_add_fwd(const void* x, const void* residual, const void* gamma,
                                 int64_t M, int64_t N, double eps, int x_dtype, int w_dtype,
                                 void* h, void* y, double* y64, float* rstd, double* rstd64) {
  if (M < 0 || N <= 0 || bad_dtypes(x_dtype, w_dtype) ||
      (M > 0 && (!x || !residual || !gamma)))
    return -1;
  double* v = (double*)malloc((size_t)N * sizeof(double));
  double* yr = (double*)malloc((size_t)N * sizeof(double));
  void* hr = malloc((size_t)N * 4);
  if (!v || !yr || !hr) { free(v); free(yr); free(hr); return -1; }
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double sum = load(residual, x_dtype, i * N + j) + load(x, x_dtype, i * N + j);
      store(hr, x_dtype, j, sum);
      v[j] = load(hr, x_dtype, j);                 /* normalise the stored h */
      if (h) store(h, x_dtype, i * N + j, sum);
    }
    double r;
    fwd_row(v, gamma, w_dtype, N, eps, &r, yr);
    if (rstd) rstd[i] = (float)r;
    if (rstd64) rstd64[i] = r;
    for (int64_t j = 0; j < N; ++j) {
      if (y) store(y, x_dtype, i * N + j, yr[j]);
      if (y64) y64[i * N + j] = yr[j];
    }
  }
  free(v);
  free(yr);
  free(hr);
  return 0;
}

/* ---- backward ------------------------------------------------------------ */

/* dy, x: M x N (x_dtype); rstd: M fp32 saved by the forward, or NULL to
 * recompute r = 1/sqrt(mean(x^2) + eps) from x; gamma: N (w_dtype).
 * Outputs (each may be NULL):
 *   dx (x_dtype, rounded once), dx64 (double) -- M x N
 *   dgamma64 (double, N), dgamma (fp32, N, rounded once from dgamma64)
 *   c64 (double, M): c of each row;  dot_abs64 (double, M): sum_k |gamma_k dy_k x_k|
 *   dgamma_sq64 (double, N): sum over rows of (dy x r)^2
 * The last three size the error of a finite-precision evaluation. */
int oracle_rmsnorm_bwd(const void* dy, const void* x, const float* rstd, const void* gamma,
                       int64_t M, int64_t N, double eps, int x_dtype, int w_dtype, void* dx,
                       double* dx64, double* dgamma64, float* dgamma, double* c64,
                       double* dot_abs64, double* dgamma_sq64) {
  if (M < 0 || N <= 0 || bad_dtypes(x_dtype, w_dtype) ||
      (M > 0 && (!dy || !x || !gamma)))
    return -1;
  double* g = (double*)malloc((size_t)N * sizeof(double));
  double* acc = (double*)calloc((size_t)N, sizeof(double));
  double* acc2 = (double*)calloc((size_t)N, sizeof(double));
  if (!g || !acc || !acc2) { free(g); free(acc); free(acc2); return -1; }
  for (int64_t j = 0; j < N; ++j) g[j] = load(gamma, w_dtype, j);
  for (int64_t i = 0; i < M; ++i) {
    double r;
    if (rstd) {
      r = (double)rstd[i];
    } else {
      double ss = 0.0;
      for (int64_t j = 0; j < N; ++j) {
        double xv = load(x, x_dtype, i * N + j);
        ss += xv * xv;
      }
      r = 1.0 / sqrt(ss / (double)N + eps);
    }
    double dot = 0.0, dabs = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      double t = g[j] * load(dy, x_dtype, i * N + j) * load(x, x_dtype, i * N + j);
      dot += t;
      dabs += fabs(t);
    }
    double c = r * r / (double)N * dot;
    if (c64) c64[i] = c;
    if (dot_abs64) dot_abs64[i] = dabs;
    for (int64_t j = 0; j < N; ++j) {
      double dyv = load(dy, x_dtype, i * N + j);
      double xv = load(x, x_dtype, i * N + j);
      double d = r * (g[j] * dyv - xv * c);
      if (dx) store(dx, x_dtype, i * N + j, d);
      if (dx64) dx64[i * N + j] = d;
      double t = dyv * xv * r;
      acc[j] += t;
      acc2[j] += t * t;
    }
  }
  for (int64_t j = 0; j < N; ++j) {
    if (dgamma64) dgamma64[j] = acc[j];
    if (dgamma) dgamma[j] = (float)acc[j];
    if (dgamma_sq64) dgamma_sq64[j] = acc2[j];
  }
  free(g);
  free(acc);
  free(acc2);
  return 0;
}

/* ---- fused residual add: backward ---------------------------------------- */

/* Backward of the fused add (the fused-add training wrapper of "Pre-built
 * kernel library guide", section 1.2, for h = residual + x, y = RMSNorm(h)):
 * h is the stored sum the forward normalised, dres the gradient that reaches
 * h along the residual path.  Both r and x receive
 *     dh = dx_rmsnorm(dy; h) + dres
 * (rounded once to x_dtype).  dgamma as in oracle_rmsnorm_bwd, and optionally
 * rounded once to w_dtype (dgamma_w).  Outputs may be NULL. */
int oracle_rmsnorm_fused_add_bwd(const void* dy, const void* h, const float* rstd,
                                 const void* gamma, const void* dres, int64_t M, int64_t N,
                                 double eps, int x_dtype, int w_dtype, void* dh, double* dh64,
                                 double* dgamma64, float* dgamma, void* dgamma_w) {
  if (M < 0 || N <= 0 || bad_dtypes(x_dtype, w_dtype) || (M > 0 && !dres)) return -1;
  double* dx64 = (double*)malloc((size_t)(M > 0 ? M : 1) * (size_t)N * sizeof(double));
  double* dg = (double*)malloc((size_t)N * sizeof(double));
  if (!dx64 || !dg) { free(dx64); free(dg); return -1; }
  int rc = oracle_rmsnorm_bwd(dy, h, rstd, gamma, M, N, eps, x_dtype, w_dtype, NULL, dx64, dg,
                              dgamma, NULL, NULL, NULL);
  if (rc == 0) {
    for (int64_t i = 0; i < M * N; ++i) {
      double v = dx64[i] + load(dres, x_dtype, i);
      if (dh) store(dh, x_dtype, i, v);
      if (dh64) dh64[i] = v;
    }
    for (int64_t j = 0; j < N; ++j) {
      if (dgamma64) dgamma64[j] = dg[j];
      if (dgamma_w) store(dgamma_w, w_dtype, j, dg[j]);
    }
  }
  free(dx64);
  free(dg);
  return rc;
}

/* ---- strided rows (per-head q/k norm) ------------------------------------ */

/* Forward over the rows of a [T, H, D] view: row (t, h) starts at element
 * t * x_st + h * x_sh of x (and t * y_st + h * y_sh of y), its D elements are
 * contiguous, and it is normalised over D with one gamma of length D shared by
 * all heads -- the per-head q/k RMSNorm of "TIRx kernels", Kernels list
 * (flashinfer.norm: qk_rmsnorm), whose rows sit inside a wider projection
 * output.  rstd (optional) is [T * H], row t * H + h.  Strides in elements. */
int oracle_rmsnorm_fwd_strided(const void* x, int64_t x_st, int64_t x_sh, const void* gamma,
                               int64_t T, int64_t H, int64_t D, double eps, int x_dtype,
                               int w_dtype, void* y, int64_t y_st, int64_t y_sh, double* y64,
                               float* rstd) {
  if (T < 0 || H < 0 || D <= 0 || bad_dtypes(x_dtype, w_dtype) ||
      (T * H > 0 && (!x || !gamma)))
    return -1;
  double* v = (double*)malloc((size_t)D * sizeof(double));
  double* yr = (double*)malloc((size_t)D * sizeof(double));
  if (!v || !yr) { free(v); free(yr); return -1; }
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t h = 0; h < H; ++h) {
      const int64_t xo = t * x_st + h * x_sh, yo = t * y_st + h * y_sh;
      for (int64_t j = 0; j < D; ++j) v[j] = load(x, x_dtype, xo + j);
      double r;
      fwd_row(v, gamma, w_dtype, D, eps, &r, yr);
      if (rstd) rstd[t * H + h] = (float)r;
      for (int64_t j = 0; j < D; ++j) {
        if (y) store(y, x_dtype, yo + j, yr[j]);
        if (y64) y64[(t * H + h) * D + j] = yr[j];
      }
    }
  }
  free(v);
  free(yr);
  return 0;
}

/* ---- quantised outputs ----------------------------------------------------- */

/* Nearest point of a small binary floating-point format to |v|, ties to the
 * even significand.  The format has `mbits` fraction bits, minimum normal
 * exponent `emin` (subnormals below 2^emin with spacing 2^(emin - mbits)) and
 * largest finite magnitude `maxv`; larger magnitudes saturate to maxv. */
static double round_small(double a, int mbits, int emin, double maxv) {
  if (a == 0.0) return 0.0;
  int k;
  frexp(a, &k);
  k -= 1;                                          /* 2^k <= a < 2^(k+1) */
  if (k < emin) k = emin;
  double ulp = ldexp(1.0, k - mbits);
  double n = a / ulp;                              /* exact: ulp is a power of two */
  double lo = floor(n), frac = n - lo, m = lo;
  if (frac > 0.5) m = lo + 1.0;
  else if (frac == 0.5) m = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
  double r = m * ulp;
  return r > maxv ? maxv : r;
}

/* Code of a magnitude that round_small returned: subnormals (below 2^emin)
 * have exponent field 0 and fraction r / 2^(emin - mbits); normals have
 * exponent field e - emin + 1 for r in [2^e, 2^(e+1)). */
static unsigned small_code(double r, int mbits, int emin) {
  if (r < ldexp(1.0, emin)) return (unsigned)(r / ldexp(1.0, emin - mbits));
  int e;
  frexp(r, &e);
  e -= 1;
  unsigned frac = (unsigned)(r / ldexp(1.0, e - mbits)) - (1u << mbits);
  return ((unsigned)(e - emin + 1) << mbits) | frac;
}

/* FP8 E4M3 (the "fn" flavour: no infinities): sign, 4 exponent bits (bias 7),
 * 3 fraction bits; normals from 2^-6 to 448 = 1.75 * 2^8, subnormals with
 * spacing 2^-9; codes 0x7F and 0xFF are NaN.  Nearest, ties to even;
 * magnitudes above 448 saturate to 448 (finite-saturating conversion);
 * NaN gives 0x7F. */
uint8_t oracle_round_e4m3(double v) {
  if (v != v) return 0x7F;
  unsigned s = signbit(v) ? 0x80u : 0u;
  double r = round_small(fabs(v), 3, -6, 448.0);
  return (uint8_t)(s | small_code(r, 3, -6));
}

double oracle_e4m3_to_double(uint8_t c) {
  unsigned e = (c >> 3) & 0xF, f = c & 7;
  if (e == 0xF && f == 7) return NAN;
  double m = e == 0 ? ldexp((double)f, -9) : ldexp(1.0 + f / 8.0, (int)e - 7);
  return (c & 0x80) ? -m : m;
}

/* FP4 E2M1: sign, 2 exponent bits (bias 1), 1 fraction bit: magnitudes 0,
 * 0.5, 1, 1.5, 2, 3, 4, 6.  Nearest, ties to the even code; magnitudes above
 * 6 saturate to 6. */
uint8_t oracle_round_e2m1(double v) {
  unsigned s = signbit(v) ? 0x8u : 0u;
  double r = round_small(fabs(v), 1, 0, 6.0);
  return (uint8_t)(s | small_code(r, 1, 0));
}

double oracle_e2m1_to_double(uint8_t c) {
  unsigned e = (c >> 1) & 3, f = c & 1;
  double m = e == 0 ? 0.5 * f : ldexp(1.0 + f / 2.0, (int)e - 1);
  return (c & 0x8) ? -m : m;
}

/* Row i of the normalised input: x, or (residual given) the stored sum
 * h = residual + x rounded to x_dtype, also written to h_out if non-NULL. */
static void quant_row_input(const void* x, const void* residual, int x_dtype, int64_t i,
                            int64_t N, void* h_out, void* hr, double* v) {
  for (int64_t j = 0; j < N; ++j) {
    if (!residual) {
      v[j] = load(x, x_dtype, i * N + j);
      continue;
    }
    double sum = load(residual, x_dtype, i * N + j) + load(x, x_dtype, i * N + j);
    store(hr, x_dtype, j, sum);
    v[j] = load(hr, x_dtype, j);
    if (h_out) store(h_out, x_dtype, i * N + j, sum);
  }
}

/* Forward with FP8 E4M3 output and one scale per row (token): the
 * quantised-output norms named in "TIRx kernels", Kernels list
 * (flashinfer.norm: rmsnorm_quant, fused_add_rmsnorm_quant).  With y the
 * forward's output (of x, or of h = residual + x when residual is given):
 *     s_i  = max_j |y_ij| / 448          (dequantisation scale, fp32)
 *     q_ij = e4m3(y_ij / s_i)            so that y_ij ~ e4m3_value(q_ij) * s_i
 * The code is decided on the fp32 value of the quotient (the exact quotient
 * rounded to fp32, then to e4m3).  A row whose x * gamma is all zero gets
 * s = 0 and q = 0 for any eps.  Outputs (each may be NULL): h (x_dtype), q
 * (M x N codes), scale (fp32) and scale64 (double), v64 (the exact quotients
 * y / s, M x N), rstd (fp32). */
int oracle_rmsnorm_fwd_fp8(const void* x, const void* residual, const void* gamma, int64_t M,
                           int64_t N, double eps, int x_dtype, int w_dtype, void* h, uint8_t* q,
                           float* scale, double* scale64, double* v64, float* rstd) {
  if (M < 0 || N <= 0 || bad_dtypes(x_dtype, w_dtype) || (M > 0 && (!x || !gamma)))
    return -1;
  double* v = (double*)malloc((size_t)N * sizeof(double));
  double* yr = (double*)malloc((size_t)N * sizeof(double));
  void* hr = malloc((size_t)N * 4);
  if (!v || !yr || !hr) { free(v); free(yr); free(hr); return -1; }
  for (int64_t i = 0; i < M; ++i) {
    quant_row_input(x, residual, x_dtype, i, N, h, hr, v);
    double r;
    fwd_row(v, gamma, w_dtype, N, eps, &r, yr);
    if (rstd) rstd[i] = (float)r;
    double m = 0.0;
    for (int64_t j = 0; j < N; ++j) m = fmax(m, fabs(v[j] * load(gamma, w_dtype, j)));
    double amax = 0.0;
    if (m > 0.0)
      for (int64_t j = 0; j < N; ++j) amax = fmax(amax, fabs(yr[j]));
    double s = amax / 448.0;
    if (scale) scale[i] = (float)s;
    if (scale64) scale64[i] = s;
    for (int64_t j = 0; j < N; ++j) {
      double quo = m > 0.0 ? yr[j] / s : 0.0;
      if (v64) v64[i * N + j] = quo;
      if (q) q[i * N + j] = oracle_round_e4m3((double)(float)quo);
    }
  }
  free(v);
  free(yr);
  free(hr);
  return 0;
}

/* Forward with NVFP4 output: the FP4 norms named in "TIRx kernels", Kernels
 * list (flashinfer.norm: rmsnorm_fp4quant, add_rmsnorm_fp4quant; the format
 * of flashinfer.quantization: nvfp4_quantize).  N is a multiple of 16 and
 * every row splits into blocks of 16 consecutive elements; gs > 0 is the
 * caller's global scale.  With y the forward's output, for block b:
 *     a_b  = max |y| over the block
 *     sf_b = e4m3(gs * a_b / 6)          S_b = its value
 *     q_j  = e2m1(y_j * gs / S_b)        (0 when S_b = 0)
 * so y_j ~ e2m1_value(q_j) * S_b / gs.  Both codes are decided on fp32
 * values (the exact value rounded to fp32, then to the small format).
 * Outputs (each may be NULL): h (x_dtype); q (M x N/2 bytes, two codes per
 * byte, element 2k in the low nibble); sf (M x N/16 codes, row-major);
 * sfv64 (the exact gs * a_b / 6, M x N/16); v64 (the exact y * gs / S_b,
 * M x N); rstd (fp32). */
int oracle_rmsnorm_fwd_nvfp4(const void* x, const void* residual, const void* gamma, int64_t M,
                             int64_t N, double eps, double gs, int x_dtype, int w_dtype, void* h,
                             uint8_t* q, uint8_t* sf, double* sfv64, double* v64, float* rstd) {
  if (M < 0 || N <= 0 || N % 16 != 0 || !(gs > 0.0) || bad_dtypes(x_dtype, w_dtype) ||
      (M > 0 && (!x || !gamma)))
    return -1;
  double* v = (double*)malloc((size_t)N * sizeof(double));
  double* yr = (double*)malloc((size_t)N * sizeof(double));
  void* hr = malloc((size_t)N * 4);
  if (!v || !yr || !hr) { free(v); free(yr); free(hr); return -1; }
  const int64_t nb = N / 16;
  for (int64_t i = 0; i < M; ++i) {
    quant_row_input(x, residual, x_dtype, i, N, h, hr, v);
    double r;
    fwd_row(v, gamma, w_dtype, N, eps, &r, yr);
    if (rstd) rstd[i] = (float)r;
    for (int64_t b = 0; b < nb; ++b) {
      double m = 0.0, a = 0.0;
      for (int64_t j = 16 * b; j < 16 * b + 16; ++j) {
        m = fmax(m, fabs(v[j] * load(gamma, w_dtype, j)));
        a = fmax(a, fabs(yr[j]));
      }
      if (m == 0.0) a = 0.0;                       /* all-zero block: a = 0 for any eps */
      double sfv = gs * a / 6.0;
      uint8_t code = oracle_round_e4m3((double)(float)sfv);
      double S = oracle_e4m3_to_double(code);
      if (sf) sf[i * nb + b] = code;
      if (sfv64) sfv64[i * nb + b] = sfv;
      for (int64_t j = 16 * b; j < 16 * b + 16; ++j) {
        double quo = S > 0.0 ? yr[j] * gs / S : 0.0;
        uint8_t c = oracle_round_e2m1((double)(float)quo);
        if (v64) v64[i * N + j] = quo;
        if (q) {
          uint8_t* byte = &q[(i * N + j) / 2];
          if (j % 2 == 0) *byte = c;
          else *byte = (uint8_t)(*byte | (c << 4));
        }
      }
    }
  }
  free(v);
  free(yr);
  free(hr);
  return 0;
}

/* ---- LayerNorm ----------------------------------------------------------- */

/* One row of LayerNorm ("Pre-built kernel library guide", section 1.1:
 * (x - mean) / sqrt(var + eps) * gamma + beta, two passes): mean, then the
 * population variance about it, each a plain double sum. */
static void ln_stats(const double* v, int64_t N, double eps, double* mean, double* rstd) {
  double s = 0.0;
  for (int64_t j = 0; j < N; ++j) s += v[j];
  const double mu = s / (double)N;
  double q = 0.0;
  for (int64_t j = 0; j < N; ++j) q += (v[j] - mu) * (v[j] - mu);
  *mean = mu;
  *rstd = 1.0 / sqrt(q / (double)N + eps);
}

/* x: M x N (x_dtype); gamma, beta: N (w_dtype; beta may be NULL for 0).
 * Outputs (each may be NULL): y (x_dtype, rounded once), y64 (double),
 * mean and rstd (fp32, rounded once), mean64 and rstd64 (double). */
int oracle_layernorm_fwd(const void* x, const void* gamma, const void* beta, int64_t M,
                         int64_t N, double eps, int x_dtype, int w_dtype, void* y, double* y64,
                         float* mean, float* rstd, double* mean64, double* rstd64) {
  if (M < 0 || N <= 0 || bad_dtypes(x_dtype, w_dtype) || (M > 0 && (!x || !gamma)))
    return -1;
  double* v = (double*)malloc((size_t)N * sizeof(double));
  if (!v) return -1;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) v[j] = load(x, x_dtype, i * N + j);
    double mu, r;
    ln_stats(v, N, eps, &mu, &r);
    if (mean) mean[i] = (float)mu;
    if (rstd) rstd[i] = (float)r;
    if (mean64) mean64[i] = mu;
    if (rstd64) rstd64[i] = r;
    for (int64_t j = 0; j < N; ++j) {
      double b = beta ? load(beta, w_dtype, j) : 0.0;
      double out = (v[j] - mu) * r * load(gamma, w_dtype, j) + b;
      if (y) store(y, x_dtype, i * N + j, out);
      if (y64) y64[i * N + j] = out;
    }
  }
  free(v);
  return 0;
}

/* Backward of the LayerNorm forward.  The pages give no formula; with
 * xhat = (x - mean) rstd and g = dy * gamma, differentiating gives
 *     dx_j     = rstd (g_j - mean_k g_k - xhat_j mean_k (g_k xhat_k))
 *     dgamma_j = sum_rows dy_j xhat_j          dbeta_j = sum_rows dy_j
 * with the saved mean and rstd (fp32, as the forward stored them) when both
 * are given, else both recomputed from x and eps.  Outputs (each may be
 * NULL): dx (x_dtype, rounded once), dx64; dgamma64, dbeta64 (double) and
 * dgamma, dbeta (fp32, rounded once); dx_scale64 (M): rstd * (sum_k |g_k| +
 * sum_k |g_k xhat_k|) / N, the size of the row terms, for error bounds. */
int oracle_layernorm_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
                         const void* gamma, int64_t M, int64_t N, double eps, int x_dtype,
                         int w_dtype, void* dx, double* dx64, double* dgamma64,
                         double* dbeta64, float* dgamma, float* dbeta, double* dx_scale64) {
  if (M < 0 || N <= 0 || bad_dtypes(x_dtype, w_dtype) || (M > 0 && (!dy || !x || !gamma)) ||
      (!mean) != (!rstd))
    return -1;
  double* v = (double*)malloc((size_t)N * sizeof(double));
  double* xh = (double*)malloc((size_t)N * sizeof(double));
  double* g = (double*)malloc((size_t)N * sizeof(double));
  double* dg = (double*)calloc((size_t)N, sizeof(double));
  double* db = (double*)calloc((size_t)N, sizeof(double));
  if (!v || !xh || !g || !dg || !db) {
    free(v); free(xh); free(g); free(dg); free(db);
    return -1;
  }
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) v[j] = load(x, x_dtype, i * N + j);
    double mu, r;
    if (mean) {
      mu = (double)mean[i];
      r = (double)rstd[i];
    } else {
      ln_stats(v, N, eps, &mu, &r);
    }
    double sg = 0.0, sgx = 0.0, ag = 0.0, agx = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      const double d = load(dy, x_dtype, i * N + j);
      xh[j] = (v[j] - mu) * r;
      g[j] = d * load(gamma, w_dtype, j);
      sg += g[j];
      sgx += g[j] * xh[j];
      ag += fabs(g[j]);
      agx += fabs(g[j] * xh[j]);
      dg[j] += d * xh[j];
      db[j] += d;
    }
    const double mg = sg / (double)N, mgx = sgx / (double)N;
    if (dx_scale64) dx_scale64[i] = r * (ag + agx) / (double)N;
    for (int64_t j = 0; j < N; ++j) {
      const double out = r * (g[j] - mg - xh[j] * mgx);
      if (dx) store(dx, x_dtype, i * N + j, out);
      if (dx64) dx64[i * N + j] = out;
    }
  }
  for (int64_t j = 0; j < N; ++j) {
    if (dgamma64) dgamma64[j] = dg[j];
    if (dbeta64) dbeta64[j] = db[j];
    if (dgamma) dgamma[j] = (float)dg[j];
    if (dbeta) dbeta[j] = (float)db[j];
  }
  free(v); free(xh); free(g); free(dg); free(db);
  return 0;
}
