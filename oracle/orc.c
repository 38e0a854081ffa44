/*
 * orc.c - float64 CPU oracle of the one-row decode MLP (test infrastructure).
 *
 * This file is TEST INFRASTRUCTURE.  Only the tests, the package's smoke check
 * and the bench's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library: it has its own bf16 rounding, its own
 * quantiser and plain loops in IEEE binary64, built with -ffp-contract=off so
 * that every operation is rounded the way it is written.
 *
 * What it computes (meTile docs):
 *  - "Compute-Graph Fusion", opening example: summed = values + residual and
 *    normalized = rms_norm(summed, weight, eps), both graph outputs.
 *  - "Compute-Graph Fusion", Automatic Gated Epilogues: two projections of one
 *    shared activation, silu(gate) * up applied before the only store, then
 *    the down projection whose epilogue adds the transformer residual.
 *  - "MLX-LM Backend", prepare/autotune section and Dispatch Policy: affine
 *    group-wise weights w = scale * q + bias with groups of 32/64/128 along K,
 *    INT8 and 4-bit "affine nibbles, scales, and biases", dense BF16 weights,
 *    and the exact "values @ weight.T + residual" down projection.
 *  - "MLX-LM Backend", the attention-projection and vocabulary compression
 *    passages before Dispatch Policy: the q/k/v/o projections of a layer and
 *    the vocabulary projection (a tied embedding used as a linear map, or an
 *    untied lm_head) run the same one-row GEMV, and the projection bias is
 *    kept: y = x @ weight.T + bias.
 *  - "MLX-LM Backend", Block-Scaled MLX Primitive: MXFP8 and MXFP4 weights,
 *    E4M3 or E2M1 element values with E8M0 block scales.  The element and
 *    scale encodings and the block size of 32 follow the OCP Microscaling
 *    Formats (MX) v1.0 specification, which the page's format names refer to.
 *  - ANEForge docs, "The optimizer and the cost model", The roofline: a weight
 *    is stored [N, K] (K contiguous) and x[.., K] @ W[N, K]^T gives [.., N].
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes of this repository):
 *  - bf16 values are rounded to nearest-even directly from binary64, only
 *    where a tensor crosses a call boundary (out_sum, out_norm, h, y).
 *  - quantiser: bias = bf16(min) (+0 for a zero minimum),
 *    scale = bf16((max - min) / (2^bits - 1)),
 *    q = clamp(round_half_even((w - bias) / scale), 0, 2^bits - 1), computed
 *    against the bf16-rounded scale and bias; a zero scale gives q = 0.
 *  - 4-bit packing: code 2j in the low nibble and code 2j+1 in the high
 *    nibble of byte j of a row.
 *  - RMSNorm: n = s * w / sqrt(mean(s^2) + eps), from the bf16-rounded sum.
 *  - SwiGLU: h = silu(g) * u with silu(g) = g / (1 + exp(-g)), no rounding
 *    of g, u or the sigmoid before h.
 *  - down: y = sum_k h_k * W[n,k] + residual_n, rounded once.
 *  - projection: y = sum_k x_k * W[n,k] + bias_n (bias bf16, absent = 0),
 *    rounded once.
 *  - MX quantiser (per block of 32 consecutive elements along K): the shared
 *    scale is 2^(floor(log2(amax)) - emax) with emax the element format's
 *    largest exponent (8 for E4M3, 2 for E2M1), its E8M0 field clamped to
 *    [0, 254] (an all-zero block takes field 0); each element is w / scale
 *    rounded to nearest-even in the element format, magnitudes above the
 *    largest finite value clamped to it, the sign kept (so a negative value
 *    that rounds to zero gives the negative-zero code).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

static uint64_t orc_bits64(double x) {
  uint64_t u;
  memcpy(&u, &x, sizeof u);
  return u;
}

/*
 * Round a binary64 value to the nearest bf16 (8 significant bits, exponent
 * range of binary32), ties to even, in one step.  Overflow gives +-inf, NaN
 * gives a quiet NaN of the same sign, subnormal bf16 results are produced
 * with their reduced precision.  The rounding is done by scaling with the
 * spacing of the target format: q = x / ulp is rounded to an integer with
 * round-half-even (nearbyint in the default rounding mode), then scaled back.
 */
uint16_t orc_bf16_from_f64(double x) {
  uint64_t u = orc_bits64(x);
  uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
  if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
  double a = fabs(x);
  if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
  int exp_unbiased = e - 1;     /* a in [2^(e-1), 2^e) */
  if (exp_unbiased < -126) exp_unbiased = -126; /* subnormal spacing */
  double ulp = ldexp(1.0, exp_unbiased - 7);
  double q = nearbyint(a / ulp); /* exact division by a power of two */
  double r = q * ulp;            /* exact */
  /* largest finite bf16 = (2 - 2^-7) * 2^127 */
  double maxf = ldexp(255.0, 120);
  if (r > maxf) return (uint16_t)(sign | 0x7F80u);
  /* encode r (a bf16 value) */
  if (r < ldexp(1.0, -126)) {   /* subnormal: r = k * 2^-133 */
    uint16_t k = (uint16_t)ldexp(r, 133);
    return (uint16_t)(sign | k);
  }
  int e2;
  double m2 = frexp(r, &e2);    /* r = m2 * 2^e2, m2 in [0.5,1) */
  int be = e2 - 1 + 127;        /* biased exponent */
  uint16_t frac = (uint16_t)(ldexp(m2, 8) - 128.0); /* 7 fraction bits */
  return (uint16_t)(sign | (uint16_t)(be << 7) | frac);
}

/* Value of a bf16 bit pattern, from its sign, exponent and fraction fields. */
double orc_f64_from_bf16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xFF;
  int f = h & 0x7F;
  double v;
  if (e == 0xFF)
    v = f ? NAN : INFINITY;
  else if (e == 0)
    v = ldexp((double)f, -133);
  else
    v = ldexp(128.0 + (double)f, e - 127 - 7);
  return sign ? -v : v;
}

void orc_bf16_from_f64_array(const double* x, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = orc_bf16_from_f64(x[i]);
}

void orc_f64_from_bf16_array(const uint16_t* h, double* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = orc_f64_from_bf16(h[i]);
}

/* ------------------------------------------------------------- quantiser */

/*
 * Affine group quantisation of W [N][K] (fp32, row-major) along K.
 * codes [N][K] (one code per byte), scales/biases [N][K/group] as bf16 bits.
 * Returns 0 on success, -1 on bad arguments.
 */
int orc_quantize(const float* W, long N, long K, int group, int bits,
                 uint8_t* codes, uint16_t* scales, uint16_t* biases) {
  if (group <= 0 || K % group != 0 || (bits != 8 && bits != 4)) return -1;
  const double qmax = (double)((1 << bits) - 1);
  const long G = K / group;
  for (long n = 0; n < N; ++n) {
    for (long gi = 0; gi < G; ++gi) {
      const float* w = W + n * K + gi * group;
      double mn = (double)w[0], mx = (double)w[0];
      for (int k = 1; k < group; ++k) {
        double v = (double)w[k];
        if (v < mn) mn = v;
        if (v > mx) mx = v;
      }
      if (mn == 0.0) mn = 0.0; /* a zero minimum gives the bias +0 */
      uint16_t b16 = orc_bf16_from_f64(mn);
      uint16_t s16 = orc_bf16_from_f64((mx - mn) / qmax);
      double bias = orc_f64_from_bf16(b16);
      double scale = orc_f64_from_bf16(s16);
      scales[n * G + gi] = s16;
      biases[n * G + gi] = b16;
      uint8_t* q = codes + n * K + gi * group;
      for (int k = 0; k < group; ++k) {
        if (scale == 0.0) {
          q[k] = 0;
          continue;
        }
        double t = nearbyint(((double)w[k] - bias) / scale);
        if (t < 0.0) t = 0.0;
        if (t > qmax) t = qmax;
        q[k] = (uint8_t)t;
      }
    }
  }
  return 0;
}

/* Stored byte layout of codes: 8 bits -> one byte per code; 4 bits -> byte j
 * of a row holds code 2j in bits 0..3 and code 2j+1 in bits 4..7. */
int orc_pack_codes(const uint8_t* codes, long N, long K, int bits, uint8_t* packed) {
  if (bits == 8) {
    memcpy(packed, codes, (size_t)(N * K));
    return 0;
  }
  if (bits != 4 || K % 2 != 0) return -1;
  for (long n = 0; n < N; ++n)
    for (long j = 0; j < K / 2; ++j) {
      uint8_t lo = codes[n * K + 2 * j], hi = codes[n * K + 2 * j + 1];
      if (lo > 15 || hi > 15) return -1;
      packed[n * (K / 2) + j] = (uint8_t)(lo | (hi << 4));
    }
  return 0;
}

/* w'[n][k] = scale * q + bias in binary64 (exact: 8-bit times 8-bit). */
int orc_dequant(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                long N, long K, int group, double* out) {
  if (group <= 0 || K % group != 0) return -1;
  const long G = K / group;
  for (long n = 0; n < N; ++n)
    for (long k = 0; k < K; ++k) {
      double s = orc_f64_from_bf16(scales[n * G + k / group]);
      double b = orc_f64_from_bf16(biases[n * G + k / group]);
      out[n * K + k] = s * (double)codes[n * K + k] + b;
    }
  return 0;
}

/* ------------------------------------------------------ weight operand */

double orc_e4m3_value(uint8_t c);
double orc_e2m1_value(uint8_t c);

/* fmt 0: dense bf16 weights [N][K]; fmt 1: affine codes [N][K] (one code per
 * byte, any bit width) with bf16 scales/biases [N][K/group]; fmt 2 / 3: MX
 * element codes [N][K] (one E4M3 / E2M1 code per byte) with E8M0 scales
 * [N][K/32] (passed as bytes through s; b unused). */
static double orc_weight(int fmt, const void* W, const uint16_t* s, const uint16_t* b,
                         long K, int group, long n, long k) {
  if (fmt == 0) return orc_f64_from_bf16(((const uint16_t*)W)[n * K + k]);
  if (fmt == 2 || fmt == 3) {
    const uint8_t c = ((const uint8_t*)W)[n * K + k];
    const uint8_t e = ((const uint8_t*)s)[n * (K / 32) + k / 32];
    const double v = fmt == 2 ? orc_e4m3_value(c) : orc_e2m1_value(c);
    return v * ldexp(1.0, (int)e - 127);
  }
  const long G = K / group;
  double sc = orc_f64_from_bf16(s[n * G + k / group]);
  double bi = orc_f64_from_bf16(b[n * G + k / group]);
  return sc * (double)((const uint8_t*)W)[n * K + k] + bi;
}

static int orc_check_fmt(int fmt, long K, int group) {
  if (fmt == 0) return 0;
  if (fmt == 2 || fmt == 3) return (group == 32 && K % 32 == 0) ? 0 : -1;
  if (fmt != 1 || group <= 0 || K % group != 0) return -1;
  return 0;
}

/* ------------------------------------------------------------------ K1 */

/*
 * out_sum[m][i]  = bf16(v + r)                                (bf16 bits)
 * out_norm[m][i] = s * w / sqrt(mean_i(s^2) + eps), s = out_sum (exact, not rounded)
 */
int orc_add_rmsnorm(const uint16_t* v, const uint16_t* r, const uint16_t* w, double eps,
                    long M, long d, uint16_t* out_sum, double* out_norm) {
  if (d <= 0) return -1;
  for (long m = 0; m < M; ++m) {
    double ss = 0.0;
    for (long i = 0; i < d; ++i) {
      uint16_t s16 = orc_bf16_from_f64(orc_f64_from_bf16(v[m * d + i]) +
                                       orc_f64_from_bf16(r[m * d + i]));
      out_sum[m * d + i] = s16;
      double s = orc_f64_from_bf16(s16);
      ss += s * s;
    }
    double denom = sqrt(ss / (double)d + eps);
    for (long i = 0; i < d; ++i) {
      double s = orc_f64_from_bf16(out_sum[m * d + i]);
      out_norm[m * d + i] = s * orc_f64_from_bf16(w[i]) / denom;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ K2 */

double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/*
 * g[m][n] = sum_k x[m][k] * Wg[n][k],  u[m][n] = sum_k x[m][k] * Wu[n][k]
 * h[m][n] = silu(g) * u  (exact, not rounded).  Optional g_out/u_out.
 * Gate and up use their own scales/biases (sg, bg) and (su, bu).
 */
int orc_swiglu_gateup(const uint16_t* x, long M, long K, long N, int fmt,
                      const void* Wg, const void* Wu,
                      const uint16_t* sg, const uint16_t* bg,
                      const uint16_t* su, const uint16_t* bu, int group,
                      double* h, double* g_out, double* u_out) {
  if (orc_check_fmt(fmt, K, group)) return -1;
  for (long m = 0; m < M; ++m)
    for (long n = 0; n < N; ++n) {
      double g = 0.0, u = 0.0;
      for (long k = 0; k < K; ++k) {
        double xv = orc_f64_from_bf16(x[m * K + k]);
        g += xv * orc_weight(fmt, Wg, sg, bg, K, group, n, k);
        u += xv * orc_weight(fmt, Wu, su, bu, K, group, n, k);
      }
      h[m * N + n] = orc_silu(g) * u;
      if (g_out) g_out[m * N + n] = g;
      if (u_out) u_out[m * N + n] = u;
    }
  return 0;
}

/* ------------------------------------------------------------------ K3 */

/* y[m][n] = sum_k h[m][k] * Wd[n][k] + res[m][n]  (exact, not rounded). */
int orc_down_residual(const uint16_t* hin, long M, long K, long N, int fmt,
                      const void* Wd, const uint16_t* s, const uint16_t* b, int group,
                      const uint16_t* res, double* y) {
  if (orc_check_fmt(fmt, K, group)) return -1;
  for (long m = 0; m < M; ++m)
    for (long n = 0; n < N; ++n) {
      double acc = 0.0;
      for (long k = 0; k < K; ++k)
        acc += orc_f64_from_bf16(hin[m * K + k]) * orc_weight(fmt, Wd, s, b, K, group, n, k);
      y[m * N + n] = acc + orc_f64_from_bf16(res[m * N + n]);
    }
  return 0;
}

/* ------------------------------------------------------- projection */

/* y[m][n] = sum_k x[m][k] * W[n][k] + bias[n]  (exact, not rounded);
 * bias is a bf16 vector [N] or NULL for a projection without bias. */
int orc_linear_bias(const uint16_t* x, long M, long K, long N, int fmt,
                    const void* W, const uint16_t* s, const uint16_t* b, int group,
                    const uint16_t* bias, double* y) {
  if (orc_check_fmt(fmt, K, group)) return -1;
  for (long m = 0; m < M; ++m)
    for (long n = 0; n < N; ++n) {
      double acc = 0.0;
      for (long k = 0; k < K; ++k)
        acc += orc_f64_from_bf16(x[m * K + k]) * orc_weight(fmt, W, s, b, K, group, n, k);
      y[m * N + n] = bias ? acc + orc_f64_from_bf16(bias[n]) : acc;
    }
  return 0;
}

/* ------------------------------------------------------ MX block scaling */

/* Value of an OCP FP8 E4M3 code: sign, 4 exponent bits (bias 7), 3 fraction
 * bits; exponent field 0 is subnormal (f * 2^-9); S.1111.111 is NaN and there
 * are no infinities. */
double orc_e4m3_value(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, f = c & 7;
  double v;
  if (e == 15 && f == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)f, -9);
  else
    v = ldexp(8.0 + (double)f, e - 7 - 3);
  return s ? -v : v;
}

/* Value of an OCP FP4 E2M1 code: sign, 2 exponent bits (bias 1), 1 fraction
 * bit; exponent field 0 is subnormal (f * 0.5). */
double orc_e2m1_value(uint8_t c) {
  const int s = (c >> 3) & 1, e = (c >> 1) & 3, f = c & 1;
  const double v = e == 0 ? 0.5 * (double)f : ldexp(2.0 + (double)f, e - 1 - 1);
  return s ? -v : v;
}

/*
 * Nearest code of a minifloat format with `mbits` fraction bits, exponent
 * bias `bias`, largest finite magnitude `maxv` and the code of that magnitude
 * `maxcode`, ties to even, magnitudes above maxv clamped to it, sign kept.
 * Same scaling method as orc_bf16_from_f64: the value divided by the format's
 * spacing at its exponent is rounded to an integer, then encoded.
 */
static uint8_t orc_minifloat(double v, int mbits, int ebits, int bias, double maxv, uint8_t maxcode) {
  const uint8_t sign = (uint8_t)(signbit(v) ? 1u << (mbits + ebits) : 0u);
  double a = fabs(v);
  if (a >= maxv) return (uint8_t)(sign | maxcode);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  int eu = e - 1;                            /* a in [2^eu, 2^(eu+1)) */
  if (eu < 1 - bias) eu = 1 - bias;          /* subnormal spacing */
  const double ulp = ldexp(1.0, eu - mbits);
  const double q = nearbyint(a / ulp);       /* exact division; ties to even */
  double r = q * ulp;
  if (r > maxv) r = maxv;                    /* cannot happen below maxv; kept for clarity */
  if (r < ldexp(1.0, 1 - bias)) {            /* subnormal (or zero): fraction = r / 2^(1-bias-mbits) */
    return (uint8_t)(sign | (uint8_t)ldexp(r, bias - 1 + mbits));
  }
  int e2;
  const double m2 = frexp(r, &e2);           /* r = m2 2^e2, m2 in [0.5, 1) */
  const int be = e2 - 1 + bias;
  const uint8_t frac = (uint8_t)(ldexp(m2, mbits + 1) - ldexp(1.0, mbits));
  return (uint8_t)(sign | (uint8_t)(be << mbits) | frac);
}

uint8_t orc_e4m3_from_f64(double v) { return orc_minifloat(v, 3, 4, 7, 448.0, 0x7E); }
uint8_t orc_e2m1_from_f64(double v) { return orc_minifloat(v, 1, 2, 1, 6.0, 0x7); }

/*
 * MX quantisation of W [N][K] (fp32) along K in blocks of 32: bits 8 gives
 * MXFP8 (E4M3 elements), bits 4 MXFP4 (E2M1).  codes [N][K] (one code per
 * byte), scales [N][K/32] as E8M0 fields.  Returns 0, or -1 on bad arguments.
 */
int orc_quantize_mx(const float* W, long N, long K, int bits, uint8_t* codes, uint8_t* scales) {
  if (K % 32 != 0 || (bits != 8 && bits != 4)) return -1;
  const int emax = bits == 8 ? 8 : 2;
  const long B = K / 32;
  for (long n = 0; n < N; ++n)
    for (long bi = 0; bi < B; ++bi) {
      const float* w = W + n * K + bi * 32;
      double amax = 0.0;
      for (int k = 0; k < 32; ++k)
        if (fabs((double)w[k]) > amax) amax = fabs((double)w[k]);
      int E = 0;
      if (amax > 0.0) {
        int e;
        frexp(amax, &e);                     /* floor(log2(amax)) = e - 1 */
        E = (e - 1) - emax + 127;
        if (E < 0) E = 0;
        if (E > 254) E = 254;
      }
      scales[n * B + bi] = (uint8_t)E;
      const double X = ldexp(1.0, E - 127);
      for (int k = 0; k < 32; ++k) {
        const double v = (double)w[k] / X;   /* exact: X is a power of two */
        codes[n * K + bi * 32 + k] = bits == 8 ? orc_e4m3_from_f64(v) : orc_e2m1_from_f64(v);
      }
    }
  return 0;
}
