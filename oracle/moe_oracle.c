/*
 * moe_oracle.c -- CPU oracle of the fused MoE layer forward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline / reference leg load this library.  The product
 * path never calls it and shares no code with it (no headers, helpers,
 * tables or constants); the only thing both sides share is the seeded input
 * generator, which holds none of the method's arithmetic.
 *
 * It is plain and slow on purpose: fp64 arithmetic, straight loops in the
 * order the definitions are written, no blocking, no fusion.  Work is split
 * over POSIX threads by independent tokens / (token, expert) pairs only.
 *
 * What it computes, and where each step is defined:
 *   RMSNorm     y_i = x_i / sqrt(mean_j x_j^2 + eps) * g_i, accumulated wide,
 *               output cast back to the input dtype (bf16)
 *                 -- "4 · La fusion de noyaux", §4.2 "Réduction + élémentaire"
 *                    (RMSNorm formula and its Triton kernel: FP32 accumulation,
 *                    cast of the result to the 16-bit type);
 *                 -- "CuTeDSL chez Perplexity", section "Norme QK" (eps inside
 *                    the reciprocal square root; result cast to x's type).
 *   Router      logits l_e = sum_j h_j Wr[e,j] (+ b_e); the k largest logits
 *               (ties to the lower expert index), softmax weights over all E
 *               experts taken at the selected ones, optionally renormalised.
 *               The pages only name the routing table ("CuTeDSL chez
 *               Perplexity", MoE dispatch/combine, "Local") and token routing
 *               (spke.com fused-MoE article, introduction); the softmax /
 *               top-k / renormalisation reading is the plain one.
 *   Align       per-expert token counts, a unique slot per token inside its
 *               expert's list, lists padded to a multiple of the tile rows
 *                 -- "CuTeDSL chez Perplexity", MoE dispatch/combine, "Local".
 *               Slots are given in ascending flat index t*k+j (a stable order
 *               in place of the pages' atomic counters).
 *   Expert MLP  SwiGLU(x) = (SiLU(x W_gate) (.) (x W_up)) W_down with gate and
 *               up concatenated into one (d x 2 d_ff) weight, gate rows first
 *                 -- "4 · La fusion de noyaux", §4.2 "GEMM + GEMM".
 *   Combine     y_t = sum_j w_tj * o_tj, accumulated in j order, cast to bf16
 *                 -- "CuTeDSL chez Perplexity", MoE dispatch/combine, "Local"
 *                    (weighted accumulation in registers into the output).
 *   MXFP8       block-scaled FP8: blocks of 32 consecutive elements along the
 *               reduction dimension share a power-of-two scale X (an E8M0 byte);
 *               each element is stored as an E4M3 code of v / X, with X chosen
 *               from the block's absolute maximum
 *                 -- "CuTeDSL chez Perplexity", "Prise en charge de Blackwell"
 *                    (MXFP8 block scaling, absolute maximum over 32 elements).
 *               The pages give no recipe for X; the plain one is the OCP
 *               Microscaling rule X = 2^(floor(log2(amax)) - 8), 8 being the
 *               largest E4M3 exponent, with codes rounded to nearest (ties to
 *               even) and clamped to +-448.  The FP8 layer quantizes the expert
 *               weights, the gathered token rows and the SwiGLU activations this
 *               way and computes everything else as the bf16 layer does.
 *   MXFP4       the same block scaling with E2M1 elements (magnitudes 0, 0.5,
 *               1, 1.5, 2, 3, 4, 6): X = 2^(floor(log2(amax)) - 2), codes rounded
 *               to nearest (ties to the even mantissa bit) and clamped to +-6
 *                 -- "CuTeDSL chez Perplexity", "Prise en charge de Blackwell"
 *                    (block-scaled 4-bit formats beside MXFP8).
 *               The FP4 layer stores only the expert weights this way; its
 *               token rows and activations are MXFP8 as above.
 *   QK-norm     per attention head of Q and of K (head_dim D elements):
 *               out_j = (w_j + weight_bias) * (x_j * rstd), rstd = 1/sqrt(mean x^2
 *               + eps), with one weight vector w[D] for all heads of Q and one for
 *               K, cast to x's type -- "CuTeDSL chez Perplexity", "Norme QK".
 *
 * The routing decision (which experts a token goes to) is an integer decided
 * by floating point, so it is taken here in the same precision the kernel
 * takes it in: fp32, with the summation order spelled out in
 * canonical_fma_sum() below.  Everything else is fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 conversions (own implementation; round to nearest, ties even)  */
/* ------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static double bf16_to_f64(uint16_t b) { return (double)bf16_to_f32(b); }

/* fp32 -> bf16, round to nearest even (finite inputs). */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* fp64 -> bf16 in ONE rounding (no intermediate fp32 rounding), ties to even. */
static uint16_t f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e;
  double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  int keep = 8;            /* significant bits of a normal bf16 */
  if (e < -125) keep = e + 133; /* subnormal: the quantum is 2^-133 */
  double q = keep < 0 ? 0.0 : nearbyint(ldexp(m, keep)); /* default mode: ties to even */
  double r = ldexp(q, e - keep);
  if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | (u >> 16));
}

/* exported for the tests' own checks of the conversions */
uint16_t oracle_f64_to_bf16(double v) { return f64_to_bf16(v); }
uint16_t oracle_f32_to_bf16(float v) { return f32_to_bf16(v); }

/* ------------------------------------------------------------------ */
/* tiny thread pool: run fn(i, ctx) for i in [0, n)                     */
/* ------------------------------------------------------------------ */

typedef void (*item_fn)(int64_t i, void* ctx);
typedef struct {
  item_fn fn;
  void* ctx;
  int64_t lo, hi;
} range_job;

static void* range_worker(void* p) {
  range_job* j = (range_job*)p;
  for (int64_t i = j->lo; i < j->hi; ++i) j->fn(i, j->ctx);
  return NULL;
}

static void parallel_for(int64_t n, int nthreads, item_fn fn, void* ctx) {
  if (n <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if (nthreads > n) nthreads = (int)n;
  range_job jobs[512];
  pthread_t tid[512];
  int started[512];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].lo = n * t / nthreads;
    jobs[t].hi = n * (t + 1) / nthreads;
    started[t] = 0;
  }
  for (int t = 1; t < nthreads; ++t) started[t] = pthread_create(&tid[t], NULL, range_worker, &jobs[t]) == 0;
  range_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (started[t])
      pthread_join(tid[t], NULL);
    else
      range_worker(&jobs[t]);
  }
}

/* ------------------------------------------------------------------ */
/* RMSNorm, fp64                                                        */
/* ------------------------------------------------------------------ */

/* One token row: rstd = 1/sqrt((1/H) sum_j x_j^2 + eps); h_j = bf16(x_j * rstd * g_j).
 * h_exact (optional) receives the unrounded fp64 values x_j * rstd * g_j. */
static void rmsnorm_row_f64(int64_t H, const uint16_t* x, const uint16_t* g, double eps,
                            uint16_t* h, double* h_exact) {
  double ss = 0.0;
  for (int64_t j = 0; j < H; ++j) {
    double xv = bf16_to_f64(x[j]);
    ss += xv * xv;
  }
  double rstd = 1.0 / sqrt(ss / (double)H + eps);
  for (int64_t j = 0; j < H; ++j) {
    double v = bf16_to_f64(x[j]) * rstd * bf16_to_f64(g[j]);
    if (h) h[j] = f64_to_bf16(v);
    if (h_exact) h_exact[j] = v;
  }
}

void oracle_rmsnorm_f64(int64_t T, int64_t H, const uint16_t* x, const uint16_t* g, double eps,
                        uint16_t* h, double* h_exact) {
  for (int64_t t = 0; t < T; ++t)
    rmsnorm_row_f64(H, x + t * H, g, eps, h ? h + t * H : NULL, h_exact ? h_exact + t * H : NULL);
}

/* ------------------------------------------------------------------ */
/* MXFP8: E4M3 codes with E8M0 block scales                             */
/* ------------------------------------------------------------------ */

/* E4M3 (bias 7, no infinities; exponent field 0: subnormal m * 2^-9): the value
 * of a code.  The codes 0x7F / 0xFF (NaN) are never produced here. */
double oracle_e4m3_decode(uint8_t c) {
  int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return sgn ? -v : v;
}

/* Nearest E4M3 code of a finite v, ties to an even mantissa, |v| > 448 -> 448. */
uint8_t oracle_e4m3_encode(double v) {
  int sgn = signbit(v) ? 1 : 0;
  double a = fabs(v);
  int e, m;
  if (a < ldexp(1.0, -6)) { /* subnormal grid: steps of 2^-9 */
    double q = nearbyint(a / ldexp(1.0, -9)); /* 0 .. 8; 8 is the smallest normal */
    if (q >= 8.0) {
      e = 1;
      m = 0;
    } else {
      e = 0;
      m = (int)q;
    }
  } else {
    int ex = (int)floor(log2(a));
    if (ldexp(1.0, ex) > a) ex -= 1; /* guard the log2 of exact powers of two */
    if (ldexp(1.0, ex + 1) <= a) ex += 1;
    double q = nearbyint(a / ldexp(1.0, ex - 3)); /* 8 .. 16 */
    if (q >= 16.0) {
      q = 8.0;
      ex += 1;
    }
    e = ex + 7;
    m = (int)q - 8;
    if (e > 15 || (e == 15 && m > 6)) { /* beyond 448: saturate */
      e = 15;
      m = 6;
    }
  }
  return (uint8_t)((sgn << 7) | (e << 3) | m);
}

/* Block exponent of 32 values with absolute maximum amax: floor(log2(amax))
 * minus the element format's largest exponent (8 for E4M3, 2 for E2M1),
 * clamped to the E8M0 range [-127, 127]; -127 for amax = 0. */
static int mx_block_exponent_of(double amax, int emax) {
  if (amax == 0.0) return -127;
  int ex = (int)floor(log2(amax));
  if (ldexp(1.0, ex) > amax) ex -= 1;
  if (ldexp(1.0, ex + 1) <= amax) ex += 1;
  ex -= emax;
  return ex < -127 ? -127 : (ex > 127 ? 127 : ex);
}

static int mx_block_exponent(double amax) { return mx_block_exponent_of(amax, 8); }

/* rows x K bf16 values (K a multiple of 32) -> codes [rows, K] and scales
 * [rows, K/32] (E8M0 bytes: exponent + 127). */
void oracle_mx_quantize(int64_t rows, int64_t K, const uint16_t* x, uint8_t* codes, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < K / 32; ++b) {
      const uint16_t* xb = x + r * K + b * 32;
      double amax = 0.0;
      for (int j = 0; j < 32; ++j) {
        double a = fabs(bf16_to_f64(xb[j]));
        if (a > amax) amax = a;
      }
      int ex = mx_block_exponent(amax);
      scales[r * (K / 32) + b] = (uint8_t)(ex + 127);
      for (int j = 0; j < 32; ++j) codes[r * K + b * 32 + j] = oracle_e4m3_encode(ldexp(bf16_to_f64(xb[j]), -ex));
    }
}

/* values of codes [rows, K] with scales [rows, K/32] */
void oracle_mx_dequantize(int64_t rows, int64_t K, const uint8_t* codes, const uint8_t* scales, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < K; ++j)
      out[r * K + j] = ldexp(oracle_e4m3_decode(codes[r * K + j]), (int)scales[r * (K / 32) + j / 32] - 127);
}

/* ------------------------------------------------------------------ */
/* MXFP4: E2M1 codes with E8M0 block scales                             */
/* ------------------------------------------------------------------ */

/* E2M1 (1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; no
 * infinities or NaN; exponent field 0: subnormal m * 0.5): the value of a
 * 4-bit code.  Magnitudes of the codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_decode(uint8_t c) {
  int e = (c >> 1) & 3, m = c & 1;
  double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (c & 8) ? -v : v;
}

/* Nearest E2M1 code of a finite v, ties to an even mantissa bit, |v| > 6 -> 6
 * (a tie always lies between neighbours of different mantissa parity). */
uint8_t oracle_e2m1_encode(double v) {
  int sgn = signbit(v) ? 1 : 0;
  double a = fabs(v);
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(a - oracle_e2m1_decode((uint8_t)c));
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return (uint8_t)((sgn << 3) | best);
}

/* rows x K bf16 values (K a multiple of 32) -> E2M1 codes [rows, K] (one per
 * byte, 0..15) and E8M0 scales [rows, K/32]: the MXFP8 rule with the E2M1
 * element format (block exponent floor(log2(amax)) - 2). */
void oracle_mx4_quantize(int64_t rows, int64_t K, const uint16_t* x, uint8_t* codes, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < K / 32; ++b) {
      const uint16_t* xb = x + r * K + b * 32;
      double amax = 0.0;
      for (int j = 0; j < 32; ++j) {
        double a = fabs(bf16_to_f64(xb[j]));
        if (a > amax) amax = a;
      }
      int ex = mx_block_exponent_of(amax, 2);
      scales[r * (K / 32) + b] = (uint8_t)(ex + 127);
      for (int j = 0; j < 32; ++j) codes[r * K + b * 32 + j] = oracle_e2m1_encode(ldexp(bf16_to_f64(xb[j]), -ex));
    }
}

/* values of E2M1 codes [rows, K] with scales [rows, K/32] */
void oracle_mx4_dequantize(int64_t rows, int64_t K, const uint8_t* codes, const uint8_t* scales, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < K; ++j)
      out[r * K + j] = ldexp(oracle_e2m1_decode(codes[r * K + j]), (int)scales[r * (K / 32) + j / 32] - 127);
}

/* ------------------------------------------------------------------ */
/* NVFP4: E2M1 codes, an E4M3 scale per 16 elements, an fp32 scale per    */
/* tensor                                                                 */
/* ------------------------------------------------------------------ */

/* Second-level (per tensor) scale of NVFP4: g = amax / (448 * 6), so that the
 * largest block scale is the largest E4M3 value; 1 for an all-zero tensor.
 * fp32, as the kernels compute it. */
static float nv4_global_of(float amax) { return amax > 0.0f ? amax / 2688.0f : 1.0f; }

/* rows x K bf16 values (K a multiple of 16) -> E2M1 codes [rows, K] (one per
 * byte), E4M3 block scales [rows, K/16] and fp32 tensor scales: one for all
 * rows (per_row 0, g_out[0]) or one per row (per_row 1, g_out[r]).  The block
 * scale and the codes are integers decided by fp32 arithmetic (the scales are
 * not powers of two), so they are taken in fp32 in the kernels' order:
 *   s_b = E4M3(amax_b / (6 g))   nearest, ties to even, saturating to 448
 *   X_b = value(s_b) * g
 *   q   = E2M1(x / X_b)          nearest, ties to even, saturating to 6; 0 where X_b = 0. */
void oracle_nv4_quantize(int64_t rows, int64_t K, const uint16_t* x, int per_row, uint8_t* codes, uint8_t* scales,
                         float* g_out) {
  float amax_t = 0.0f;
  if (!per_row) {
    for (int64_t i = 0; i < rows * K; ++i) {
      float a = fabsf(bf16_to_f32(x[i]));
      if (a > amax_t) amax_t = a;
    }
    g_out[0] = nv4_global_of(amax_t);
  }
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * K;
    float g;
    if (per_row) {
      float amax_r = 0.0f;
      for (int64_t j = 0; j < K; ++j) {
        float a = fabsf(bf16_to_f32(xr[j]));
        if (a > amax_r) amax_r = a;
      }
      g = nv4_global_of(amax_r);
      g_out[r] = g;
    } else {
      g = g_out[0];
    }
    const float six_g = 6.0f * g;
    for (int64_t b = 0; b < K / 16; ++b) {
      float amax_b = 0.0f;
      for (int j = 0; j < 16; ++j) {
        float a = fabsf(bf16_to_f32(xr[b * 16 + j]));
        if (a > amax_b) amax_b = a;
      }
      const float u = amax_b / six_g;
      const uint8_t sc = oracle_e4m3_encode((double)u);
      scales[r * (K / 16) + b] = sc;
      const float X = (float)oracle_e4m3_decode(sc) * g;
      for (int j = 0; j < 16; ++j) {
        const float v = bf16_to_f32(xr[b * 16 + j]);
        codes[r * K + b * 16 + j] = X > 0.0f ? oracle_e2m1_encode((double)(v / X)) : 0;
      }
    }
  }
}

/* values of NVFP4 codes [rows, K] with block scales [rows, K/16] and tensor
 * scales g (g[0] for all rows, or g[r] per row): q * value(s) * g, in fp64 */
void oracle_nv4_dequantize(int64_t rows, int64_t K, const uint8_t* codes, const uint8_t* scales, const float* g,
                           int per_row, double* out) {
  for (int64_t r = 0; r < rows; ++r) {
    const double gr = (double)(per_row ? g[r] : g[0]);
    for (int64_t j = 0; j < K; ++j)
      out[r * K + j] = oracle_e2m1_decode(codes[r * K + j]) * oracle_e4m3_decode(scales[r * (K / 16) + j / 16]) * gr;
  }
}

/* weight rows of the low-precision layers: E4M3 (wfmt 0) or E2M1 (wfmt 1) codes
 * with E8M0 scales per 32; NVFP4 (wfmt 2): E2M1 codes, E4M3 scales per 16 and the
 * matrix's tensor scale g */
static void mx_weight_dequantize(int wfmt, int64_t rows, int64_t K, const uint8_t* codes, const uint8_t* scales,
                                 float g, double* out) {
  if (wfmt == 2)
    oracle_nv4_dequantize(rows, K, codes, scales, &g, 0, out);
  else if (wfmt)
    oracle_mx4_dequantize(rows, K, codes, scales, out);
  else
    oracle_mx_dequantize(rows, K, codes, scales, out);
}

/* one row of K bf16 token values through MXFP8 (afmt 0), MXFP4 (afmt 1) or
 * NVFP4 with a per-row tensor scale (afmt 2) quantization and back */
static void mx_token_roundtrip(int afmt, int64_t K, const uint16_t* x16, double* out) {
  uint8_t* c = (uint8_t*)malloc((size_t)K);
  uint8_t* sc = (uint8_t*)malloc((size_t)(K / 16));
  if (afmt == 2) {  /* NVFP4 with the row as the tensor */
    float g;
    oracle_nv4_quantize(1, K, x16, 1, c, sc, &g);
    oracle_nv4_dequantize(1, K, c, sc, &g, 1, out);
  } else if (afmt) {
    oracle_mx4_quantize(1, K, x16, c, sc);
    oracle_mx4_dequantize(1, K, c, sc, out);
  } else {
    oracle_mx_quantize(1, K, x16, c, sc);
    oracle_mx_dequantize(1, K, c, sc, out);
  }
  free(c);
  free(sc);
}

/* ------------------------------------------------------------------ */
/* QK-norm, fp64                                                        */
/* ------------------------------------------------------------------ */

/* rows head vectors of D elements each (a row = one head of one token):
 * rstd = 1/sqrt((1/D) sum_j x_j^2 + eps); out_j = bf16((w_j + weight_bias) * (x_j * rstd)). */
void oracle_qk_norm_f64(int64_t rows, int64_t D, const uint16_t* x, const uint16_t* w, double weight_bias,
                        double eps, uint16_t* out) {
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * D;
    double ss = 0.0;
    for (int64_t j = 0; j < D; ++j) {
      double xv = bf16_to_f64(xr[j]);
      ss += xv * xv;
    }
    double rstd = 1.0 / sqrt(ss / (double)D + eps);
    for (int64_t j = 0; j < D; ++j)
      out[r * D + j] = f64_to_bf16((bf16_to_f64(w[j]) + weight_bias) * (bf16_to_f64(xr[j]) * rstd));
  }
}

/* ------------------------------------------------------------------ */
/* Router logits, fp64                                                  */
/* ------------------------------------------------------------------ */

static void router_row_f64(int64_t H, int64_t E, const uint16_t* h, const float* Wr, const float* bias,
                           double* logits) {
  for (int64_t e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int64_t j = 0; j < H; ++j) acc += bf16_to_f64(h[j]) * (double)Wr[e * H + j];
    logits[e] = acc + (bias ? (double)bias[e] : 0.0);
  }
}

void oracle_router_logits_f64(int64_t T, int64_t H, int64_t E, const uint16_t* h, const float* Wr,
                              const float* bias, double* logits) {
  for (int64_t t = 0; t < T; ++t) router_row_f64(H, E, h + t * H, Wr, bias, logits + t * E);
}

/* ------------------------------------------------------------------ */
/* fp32 routing in the canonical summation order                        */
/* ------------------------------------------------------------------ */

/* Sum of a_j*b_j over j < H in fp32, in this fixed order:
 *   the H products are cut into chunks of 8 consecutive elements; chunk c
 *   belongs to lane c mod 32 (32 lanes); each lane accumulates its chunks in
 *   increasing c and, inside a chunk, in increasing j, each step one fused
 *   multiply-add acc = fma(a_j, b_j, acc) starting from +0;
 *   the 32 lane sums are then combined by an xor butterfly: for off = 16, 8,
 *   4, 2, 1 every lane L takes s_L + s_(L xor off).  The result is lane 0's. */
static float canonical_fma_sum(int64_t H, const float* a, const float* b) {
  float s[32];
  for (int L = 0; L < 32; ++L) {
    float acc = 0.0f;
    for (int64_t c = L; c * 8 < H; c += 32)
      for (int64_t j = c * 8; j < c * 8 + 8 && j < H; ++j) acc = fmaf(a[j], b[j], acc);
    s[L] = acc;
  }
  for (int off = 16; off >= 1; off >>= 1) {
    float nxt[32];
    for (int L = 0; L < 32; ++L) nxt[L] = s[L] + s[L ^ off];
    memcpy(s, nxt, sizeof(nxt));
  }
  return s[0];
}

typedef struct {
  int64_t H, E;
  const uint16_t *x, *g;
  float eps;
  const float *Wr, *bias;
  uint16_t* h32;
  float* logits32;
  float* rstd32;
} route32_ctx;

static void route32_token(int64_t t, void* p) {
  route32_ctx* c = (route32_ctx*)p;
  int64_t H = c->H;
  float* xs = (float*)malloc(sizeof(float) * (size_t)H);
  float* hs = (float*)malloc(sizeof(float) * (size_t)H);
  for (int64_t j = 0; j < H; ++j) xs[j] = bf16_to_f32(c->x[t * H + j]);
  float ss = canonical_fma_sum(H, xs, xs);
  float ms = ss / (float)H;
  float rstd = 1.0f / sqrtf(ms + c->eps);
  if (c->rstd32) c->rstd32[t] = rstd;
  for (int64_t j = 0; j < H; ++j) {
    float v = xs[j] * rstd;
    v = v * bf16_to_f32(c->g[j]);
    uint16_t hb = f32_to_bf16(v);
    if (c->h32) c->h32[t * H + j] = hb;
    hs[j] = bf16_to_f32(hb);
  }
  for (int64_t e = 0; e < c->E; ++e) {
    float l = canonical_fma_sum(H, hs, c->Wr + e * H);
    if (c->bias) l = l + c->bias[e];
    c->logits32[t * c->E + e] = l;
  }
  free(xs);
  free(hs);
}

/* The kernel-precision routing front end: RMSNorm in fp32 (sum of squares in
 * canonical order, mean by fp32 division, rstd = 1/sqrt(mean + eps) with IEEE
 * sqrt and division), h = bf16((x*rstd)*g), then fp32 logits in canonical
 * order plus the fp32 bias. */
void oracle_route_f32(int64_t T, int64_t H, int64_t E, const uint16_t* x, const uint16_t* g, float eps,
                      const float* Wr, const float* bias, uint16_t* h32, float* logits32, float* rstd32,
                      int nthreads) {
  route32_ctx c = {H, E, x, g, eps, Wr, bias, h32, logits32, rstd32};
  parallel_for(T, nthreads, route32_token, &c);
}

/* ------------------------------------------------------------------ */
/* top-k selection and routing weights                                   */
/* ------------------------------------------------------------------ */

/* k largest of E values, largest first; equal values: lower index first. */
void oracle_topk_f32(int64_t T, int64_t E, int k, const float* logits, int32_t* ids) {
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      ids[t * k + j] = (int32_t)best;
    }
  }
  free(taken);
}

void oracle_topk_f64(int64_t T, int64_t E, int k, const double* logits, int32_t* ids) {
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      ids[t * k + j] = (int32_t)best;
    }
  }
  free(taken);
}

/* w_j = softmax(l)[ids_j] over all E experts; with renorm, divided by the sum
 * over the k selected (which equals a softmax over the selected logits). */
void oracle_route_weights_f64(int64_t T, int64_t E, int k, const double* logits, const int32_t* ids,
                              int renorm, double* w) {
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    double m = l[0];
    for (int64_t e = 1; e < E; ++e)
      if (l[e] > m) m = l[e];
    double z = 0.0;
    for (int64_t e = 0; e < E; ++e) z += exp(l[e] - m);
    double s = 0.0;
    for (int j = 0; j < k; ++j) {
      w[t * k + j] = exp(l[ids[t * k + j]] - m) / z;
      s += w[t * k + j];
    }
    if (renorm)
      for (int j = 0; j < k; ++j) w[t * k + j] /= s;
  }
}

/* ------------------------------------------------------------------ */
/* expert align                                                          */
/* ------------------------------------------------------------------ */

/* N = T*k routing entries (flat index i = t*k + j, expert ids[i]).
 * counts[e]     number of entries routed to e
 * offsets[e]    start of e's list; lists are padded to a multiple of `pad`
 *               rows (an empty list takes no rows); offsets[E] = total rows
 * sorted_ids[p] the flat index stored in row p, entries of one expert in
 *               increasing flat index; padding rows hold the sentinel N
 * slot_of[i]    the row of entry i (inverse of sorted_ids on real rows)
 * Returns the total row count, or -1 if it exceeds `cap`. */
int64_t oracle_align(int64_t N, int64_t E, const int32_t* ids, int64_t pad, int32_t* counts,
                     int32_t* offsets, int32_t* sorted_ids, int64_t cap, int32_t* slot_of) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < N; ++i) counts[ids[i]] += 1;
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) {
    int64_t padded = (counts[e] + pad - 1) / pad * pad;
    offsets[e + 1] = (int32_t)(offsets[e] + padded);
  }
  int64_t total = offsets[E];
  if (total > cap) return -1;
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t i = 0; i < N; ++i) {
    int32_t e = ids[i];
    sorted_ids[cursor[e]] = (int32_t)i;
    slot_of[i] = cursor[e];
    cursor[e] += 1;
  }
  for (int64_t e = 0; e < E; ++e)
    for (int64_t p = offsets[e] + counts[e]; p < offsets[e + 1]; ++p) sorted_ids[p] = (int32_t)N;
  free(cursor);
  return total;
}

/* ------------------------------------------------------------------ */
/* expert MLP (SwiGLU), fp64                                             */
/* ------------------------------------------------------------------ */

/* One token through one expert.
 *   gate_i = sum_j h_j W13[i, j]        (rows [0, I) of W13[e])
 *   up_i   = sum_j h_j W13[I + i, j]    (rows [I, 2I) of W13[e])
 *   a_i    = SiLU(gate_i) * up_i,  SiLU(z) = z / (1 + e^-z); bf16-rounded if round_act
 *   o_n    = sum_i a_i W2[n, i]
 * h is given either as bf16 bits (h16) or as fp64 values (h64). */
static void expert_row_f64(int64_t H, int64_t I, const uint16_t* h16, const double* h64,
                           const uint16_t* W13e, const uint16_t* W2e, int round_act, double* a, double* o) {
  for (int64_t i = 0; i < I; ++i) {
    double gate = 0.0, up = 0.0;
    const uint16_t* wg = W13e + i * H;
    const uint16_t* wu = W13e + (I + i) * H;
    for (int64_t j = 0; j < H; ++j) {
      double hv = h16 ? bf16_to_f64(h16[j]) : h64[j];
      gate += hv * bf16_to_f64(wg[j]);
      up += hv * bf16_to_f64(wu[j]);
    }
    double silu = gate / (1.0 + exp(-gate));
    double v = silu * up;
    a[i] = round_act ? bf16_to_f64(f64_to_bf16(v)) : v;
  }
  for (int64_t n = 0; n < H; ++n) {
    double acc = 0.0;
    const uint16_t* wd = W2e + n * I;
    for (int64_t i = 0; i < I; ++i) acc += a[i] * bf16_to_f64(wd[i]);
    o[n] = acc;
  }
}

/* One token through one expert of the block-scaled layers: h (bf16) quantized
 * along H to MXFP8 (afmt 0) or MXFP4 (afmt 1), the weights given as MXFP8
 * codes and scales (wfmt 0) or MXFP4 codes (wfmt 1, E2M1, one per byte), the
 * bf16 SwiGLU activation quantized along I in the token format; products and
 * sums in fp64.
 *   W13c [2I, H] codes, W13s [2I, H/32] scales; W2c [H, I], W2s [H, I/32]. */
static void expert_row_mx_f64(int wfmt, int afmt, int64_t H, int64_t I, const uint16_t* h16, const uint8_t* W13c,
                              const uint8_t* W13s, float g13, const uint8_t* W2c, const uint8_t* W2s, float g2,
                              double* a, double* o) {
  const int64_t bs = wfmt == 2 ? 16 : 32;  /* elements per scale */
  double* hq = (double*)malloc(sizeof(double) * (size_t)H);
  mx_token_roundtrip(afmt, H, h16, hq);
  double* wrow = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
  double* wrow2 = (double*)malloc(sizeof(double) * (size_t)H);
  uint16_t* a16 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
  for (int64_t i = 0; i < I; ++i) {
    mx_weight_dequantize(wfmt, 1, H, W13c + i * H, W13s + i * (H / bs), g13, wrow);
    mx_weight_dequantize(wfmt, 1, H, W13c + (I + i) * H, W13s + (I + i) * (H / bs), g13, wrow2);
    double gate = 0.0, up = 0.0;
    for (int64_t j = 0; j < H; ++j) {
      gate += hq[j] * wrow[j];
      up += hq[j] * wrow2[j];
    }
    double silu = gate / (1.0 + exp(-gate));
    a16[i] = f64_to_bf16(silu * up);
  }
  mx_token_roundtrip(afmt, I, a16, a);
  for (int64_t n = 0; n < H; ++n) {
    mx_weight_dequantize(wfmt, 1, I, W2c + n * I, W2s + n * (I / bs), g2, wrow);
    double acc = 0.0;
    for (int64_t i = 0; i < I; ++i) acc += a[i] * wrow[i];
    o[n] = acc;
  }
  free(hq); free(wrow); free(wrow2); free(a16);
}

void oracle_expert_mx_f64(int64_t H, int64_t I, const uint16_t* h16, const uint8_t* W13c, const uint8_t* W13s,
                          const uint8_t* W2c, const uint8_t* W2s, double* a_out, double* o) {
  double* a = a_out ? a_out : (double*)malloc(sizeof(double) * (size_t)I);
  expert_row_mx_f64(0, 0, H, I, h16, W13c, W13s, 1.0f, W2c, W2s, 1.0f, a, o);
  if (!a_out) free(a);
}

/* the same with MXFP4 weights (E2M1 codes, one per byte) */
void oracle_expert_mx4_f64(int64_t H, int64_t I, const uint16_t* h16, const uint8_t* W13c, const uint8_t* W13s,
                           const uint8_t* W2c, const uint8_t* W2s, double* a_out, double* o) {
  double* a = a_out ? a_out : (double*)malloc(sizeof(double) * (size_t)I);
  expert_row_mx_f64(1, 0, H, I, h16, W13c, W13s, 1.0f, W2c, W2s, 1.0f, a, o);
  if (!a_out) free(a);
}

void oracle_expert_f64(int64_t H, int64_t I, const uint16_t* h16, const double* h64, const uint16_t* W13e,
                       const uint16_t* W2e, int round_act, double* a_out, double* o) {
  double* a = a_out ? a_out : (double*)malloc(sizeof(double) * (size_t)I);
  expert_row_f64(H, I, h16, h64, W13e, W2e, round_act, a, o);
  if (!a_out) free(a);
}

/* ------------------------------------------------------------------ */
/* the whole layer for a sample of tokens                                */
/* ------------------------------------------------------------------ */

typedef struct {
  int64_t T, H, I, E;
  int k, renorm, round_inter;
  double eps;
  const uint16_t *x, *g;
  const float *Wr, *bias;
  const uint16_t *W13, *W2;
  /* block-scaled layers (when W13c != NULL): MXFP8 weights (wfmt 0) or MXFP4
   * weights (wfmt 1); MXFP8 (afmt 0) or MXFP4 (afmt 1) tokens and activations */
  const uint8_t *W13c, *W13s, *W2c, *W2s;
  const float *W13g, *W2g; /* NVFP4: tensor scale per expert matrix */
  int wfmt, afmt;
  int64_t ns;
  const int64_t* sample;
  /* per-sample scratch / outputs */
  uint16_t* h16;   /* [ns, H] */
  double* h64;     /* [ns, H] */
  double* l64;     /* [ns, E] */
  float* l32;      /* [ns, E] */
  int32_t* ids;    /* [ns, k] */
  double* w;       /* [ns, k] */
  double* o;       /* [ns, k, H] */
} fwd_ctx;

static void fwd_route_token(int64_t s, void* p) {
  fwd_ctx* c = (fwd_ctx*)p;
  int64_t t = c->sample ? c->sample[s] : s;
  const uint16_t* xr = c->x + t * c->H;
  rmsnorm_row_f64(c->H, xr, c->g, c->eps, c->h16 + s * c->H, c->h64 + s * c->H);
  router_row_f64(c->H, c->E, c->h16 + s * c->H, c->Wr, c->bias, c->l64 + s * c->E);
  /* the routing decision in the kernel's precision */
  route32_ctx r = {c->H, c->E, xr, c->g, (float)c->eps, c->Wr, c->bias, NULL, c->l32 + s * c->E, NULL};
  route32_token(0, &r);
  oracle_topk_f32(1, c->E, c->k, c->l32 + s * c->E, c->ids + s * c->k);
  oracle_route_weights_f64(1, c->E, c->k, c->l64 + s * c->E, c->ids + s * c->k, c->renorm, c->w + s * c->k);
}

static void fwd_expert_item(int64_t it, void* p) {
  fwd_ctx* c = (fwd_ctx*)p;
  int64_t s = it / c->k;
  int j = (int)(it % c->k);
  int64_t e = c->ids[s * c->k + j];
  double* a = (double*)malloc(sizeof(double) * (size_t)c->I);
  if (c->W13c) {
    const int64_t bs = c->wfmt == 2 ? 16 : 32;
    expert_row_mx_f64(c->wfmt, c->afmt, c->H, c->I, c->h16 + s * c->H, c->W13c + e * 2 * c->I * c->H,
                      c->W13s + e * 2 * c->I * (c->H / bs), c->W13g ? c->W13g[e] : 1.0f, c->W2c + e * c->H * c->I,
                      c->W2s + e * c->H * (c->I / bs), c->W2g ? c->W2g[e] : 1.0f, a, c->o + it * c->H);
    free(a);
    return;
  }
  const uint16_t* W13e = c->W13 + e * 2 * c->I * c->H;
  const uint16_t* W2e = c->W2 + e * c->H * c->I;
  if (c->round_inter)
    expert_row_f64(c->H, c->I, c->h16 + s * c->H, NULL, W13e, W2e, 1, a, c->o + it * c->H);
  else
    expert_row_f64(c->H, c->I, NULL, c->h64 + s * c->H, W13e, W2e, 0, a, c->o + it * c->H);
  free(a);
}

/* Layer forward for ns tokens (sample[s] = token index, or sample = NULL for
 * tokens 0..ns-1).  Outputs per sampled token: the selected experts ids[s,k]
 * (decided in fp32, see oracle_route_f32), their fp64 weights w[s,k], the
 * fp64 output y64[s,H] and its bf16 rounding y16[s,H].  Optional: h16[s,H]
 * (fp64-path norm output), l32[s,E] (fp32 canonical logits), l64[s,E].
 * round_inter = 1 rounds h and the SwiGLU output to bf16 (the layer's storage
 * types); 0 keeps them in fp64 ("pure" mode).  Returns 0, or -1 on bad input. */
static int moe_forward_any(int64_t T, int64_t H, int64_t I, int64_t E, int k, int renorm, double eps,
                           const uint16_t* x, const uint16_t* g, const float* Wr, const float* bias,
                           const uint16_t* W13, const uint16_t* W2, const uint8_t* W13c, const uint8_t* W13s,
                           const uint8_t* W2c, const uint8_t* W2s, const float* W13g, const float* W2g, int wfmt,
                           int afmt, int64_t ns, const int64_t* sample,
                           int round_inter, int nthreads, int32_t* ids, double* w, double* y64, uint16_t* y16,
                           uint16_t* h16_out, float* l32_out, double* l64_out) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E || ns < 0) return -1;
  for (int64_t s = 0; s < ns; ++s) {
    int64_t t = sample ? sample[s] : s;
    if (t < 0 || t >= T) return -1;
  }
  if (ns == 0) return 0;
  fwd_ctx c;
  c.T = T; c.H = H; c.I = I; c.E = E; c.k = k; c.renorm = renorm; c.round_inter = round_inter;
  c.eps = eps; c.x = x; c.g = g; c.Wr = Wr; c.bias = bias; c.W13 = W13; c.W2 = W2;
  c.W13c = W13c; c.W13s = W13s; c.W2c = W2c; c.W2s = W2s; c.wfmt = wfmt; c.afmt = afmt;
  c.W13g = W13g; c.W2g = W2g;
  c.ns = ns; c.sample = sample;
  c.h16 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(ns * H));
  c.h64 = (double*)malloc(sizeof(double) * (size_t)(ns * H));
  c.l64 = (double*)malloc(sizeof(double) * (size_t)(ns * E));
  c.l32 = (float*)malloc(sizeof(float) * (size_t)(ns * E));
  c.ids = ids;
  c.w = w;
  c.o = (double*)malloc(sizeof(double) * (size_t)(ns * k * H));
  parallel_for(ns, nthreads, fwd_route_token, &c);
  parallel_for(ns * k, nthreads, fwd_expert_item, &c);
  for (int64_t s = 0; s < ns; ++s) {
    for (int64_t n = 0; n < H; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += w[s * k + j] * c.o[(s * k + j) * H + n];
      y64[s * H + n] = acc;
      if (y16) y16[s * H + n] = f64_to_bf16(acc);
    }
  }
  if (h16_out) memcpy(h16_out, c.h16, sizeof(uint16_t) * (size_t)(ns * H));
  if (l32_out) memcpy(l32_out, c.l32, sizeof(float) * (size_t)(ns * E));
  if (l64_out) memcpy(l64_out, c.l64, sizeof(double) * (size_t)(ns * E));
  free(c.h16); free(c.h64); free(c.l64); free(c.l32); free(c.o);
  return 0;
}

int oracle_moe_forward(int64_t T, int64_t H, int64_t I, int64_t E, int k, int renorm, double eps,
                       const uint16_t* x, const uint16_t* g, const float* Wr, const float* bias,
                       const uint16_t* W13, const uint16_t* W2, int64_t ns, const int64_t* sample,
                       int round_inter, int nthreads, int32_t* ids, double* w, double* y64, uint16_t* y16,
                       uint16_t* h16_out, float* l32_out, double* l64_out) {
  return moe_forward_any(T, H, I, E, k, renorm, eps, x, g, Wr, bias, W13, W2, NULL, NULL, NULL, NULL, NULL, NULL, 0,
                         0, ns, sample, round_inter, nthreads, ids, w, y64, y16, h16_out, l32_out, l64_out);
}

/* The FP8 layer: the same routing; the experts with MXFP8 weights (codes and
 * scales per expert as in expert_row_mx_f64, experts stacked) and MXFP8
 * activations.  H and I multiples of 32. */
int oracle_moe_forward_mx(int64_t T, int64_t H, int64_t I, int64_t E, int k, int renorm, double eps,
                          const uint16_t* x, const uint16_t* g, const float* Wr, const float* bias,
                          const uint8_t* W13c, const uint8_t* W13s, const uint8_t* W2c, const uint8_t* W2s,
                          int64_t ns, const int64_t* sample, int nthreads, int32_t* ids, double* w, double* y64,
                          uint16_t* y16) {
  if (H % 32 || I % 32 || !W13c || !W13s || !W2c || !W2s) return -1;
  return moe_forward_any(T, H, I, E, k, renorm, eps, x, g, Wr, bias, NULL, NULL, W13c, W13s, W2c, W2s, NULL, NULL,
                         0, 0, ns, sample, 1, nthreads, ids, w, y64, y16, NULL, NULL, NULL);
}

/* The FP4-weight layer: as oracle_moe_forward_mx with MXFP4 expert weights
 * (E2M1 codes, one per byte, and E8M0 scales), MXFP8 tokens and activations. */
int oracle_moe_forward_mx4(int64_t T, int64_t H, int64_t I, int64_t E, int k, int renorm, double eps,
                           const uint16_t* x, const uint16_t* g, const float* Wr, const float* bias,
                           const uint8_t* W13c, const uint8_t* W13s, const uint8_t* W2c, const uint8_t* W2s,
                           int64_t ns, const int64_t* sample, int nthreads, int32_t* ids, double* w, double* y64,
                           uint16_t* y16) {
  if (H % 32 || I % 32 || !W13c || !W13s || !W2c || !W2s) return -1;
  return moe_forward_any(T, H, I, E, k, renorm, eps, x, g, Wr, bias, NULL, NULL, W13c, W13s, W2c, W2s, NULL, NULL,
                         1, 0, ns, sample, 1, nthreads, ids, w, y64, y16, NULL, NULL, NULL);
}

/* The MXFP4 layer: MXFP4 expert weights and MXFP4 tokens and activations
 * (h and the SwiGLU activation quantized to E2M1 codes with E8M0 scales per 32
 * elements), otherwise as oracle_moe_forward_mx. */
int oracle_moe_forward_mx4a4(int64_t T, int64_t H, int64_t I, int64_t E, int k, int renorm, double eps,
                             const uint16_t* x, const uint16_t* g, const float* Wr, const float* bias,
                             const uint8_t* W13c, const uint8_t* W13s, const uint8_t* W2c, const uint8_t* W2s,
                             int64_t ns, const int64_t* sample, int nthreads, int32_t* ids, double* w, double* y64,
                             uint16_t* y16) {
  if (H % 32 || I % 32 || !W13c || !W13s || !W2c || !W2s) return -1;
  return moe_forward_any(T, H, I, E, k, renorm, eps, x, g, Wr, bias, NULL, NULL, W13c, W13s, W2c, W2s, NULL, NULL,
                         1, 1, ns, sample, 1, nthreads, ids, w, y64, y16, NULL, NULL, NULL);
}

/* The NVFP4 layer: NVFP4 expert weights (E2M1 codes [E, rows, K] one per
 * byte, E4M3 scales [E, rows, K/16], tensor scales W13g[E], W2g[E]: one per
 * expert matrix) and NVFP4 tokens and activations (one tensor scale per row),
 * otherwise as oracle_moe_forward_mx.  H and I multiples of 16. */
int oracle_moe_forward_nv4(int64_t T, int64_t H, int64_t I, int64_t E, int k, int renorm, double eps,
                           const uint16_t* x, const uint16_t* g, const float* Wr, const float* bias,
                           const uint8_t* W13c, const uint8_t* W13s, const float* W13g, const uint8_t* W2c,
                           const uint8_t* W2s, const float* W2g, int64_t ns, const int64_t* sample, int nthreads,
                           int32_t* ids, double* w, double* y64, uint16_t* y16) {
  if (H % 16 || I % 16 || !W13c || !W13s || !W13g || !W2c || !W2s || !W2g) return -1;
  return moe_forward_any(T, H, I, E, k, renorm, eps, x, g, Wr, bias, NULL, NULL, W13c, W13s, W2c, W2s, W13g, W2g, 2,
                         2, ns, sample, 1, nthreads, ids, w, y64, y16, NULL, NULL, NULL);
}

int oracle_version(void) { return 5; }
