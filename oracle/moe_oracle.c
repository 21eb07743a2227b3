/*
 * moe_oracle.c -- plain, slow, deliberately obvious CPU oracle for the
 * block-scaled MoE top-k expert layer (A8W4 and A4W4).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library in block_scaled_moe_topk_gb300/.
 *
 * What it computes, step by step, in the order of the method:
 *
 *  1. Top-k softmax gating ("[HIP] gfx950 A8W4 fused_moe configs for DSv4.1
 *     TP-sharded experts", Changes: csrc/kernels/topk_softmax_kernels.cu):
 *     experts ranked by fp32 logit, descending, ties to the lower index;
 *     softmax in double; the k selected probabilities renormalised to sum 1.
 *  2. Stable counting sort of the (token, slot) pairs by expert -- the local
 *     form of the dispatch step of "feat(moe): FlyDSL MegaMoE fused EP-MoE
 *     integration" (description: the expert step is dispatch, GEMM1, quant,
 *     GEMM2, combine), with 64-bit offsets (the same page reports an int32
 *     kernel argument overflowing on larger batches).
 *  3. MX quantisation of BF16 activations with one E8M0 scale per 1x32 block
 *     ("add A4W4 and FP8 P2P transport support to MegaMoE", Technical
 *     Details: BF16 activations become MXFP4 codes with a per-1x32 E8M0
 *     scale; the same with FP8 E4M3 codes for A8W4).  Element formats and
 *     the scale rule follow the OCP Microscaling (MX) v1.0 definitions:
 *     X = 2^(floor(log2 amax) - emax_elem), codes = RNE-satfinite(v / X).
 *  4. GEMM1 against gate/up-interleaved MXFP4 weights (row 2j = gate_j,
 *     row 2j+1 = up_j: "feat(moe): FlyDSL MegaMoE ..." description, the
 *     INTERLEAVE(g1u1) gate mode), products of decoded codes summed in
 *     double, rounded once to fp32.
 *  5. SwiGLU h_j = silu(gate_j) * up_j in fp32.  With the bf16-h option
 *     (ORACLE_OPT_H_BF16) h is rounded to bf16 first: the bf16-out stage-1
 *     family of "[HIP] gfx950 A8W4 fused_moe configs for DSv4.1 TP-sharded
 *     experts" (How the rows were chosen), whose GEMM1 writes bf16 and a
 *     separate kernel requantises.
 *  6. Requantisation of h to MX (A2: the same page on MegaMoE has the A4W4
 *     stage 1 produce FP4 A2 codes with their scales; MXFP8 for A8W4).
 *  7. GEMM2 (same arithmetic as 4).
 *  8. Top-k-weighted combine, accumulated in slot order (the pages sum the
 *     top-k contributions in FP32; the oracle uses fp64), rounded once to
 *     bf16 (round to nearest even).
 *
 * Readings where the pages are silent (all listed in the design notes):
 *  - amax == 0 or fp32-subnormal: scale byte 0, every code a signed zero.
 *  - a negative value that rounds to zero keeps its sign (E4M3 0x80, E2M1 0x8).
 *  - FP4 packing: element 2i in the low nibble of byte i, 2i+1 in the high.
 *  - E8M0 scales row-major [rows, K/32].
 *  - h is quantised from fp32 (never rounded to bf16 first); no SwiGLU clamp.
 *  - the top-k weights scale the fp32 GEMM2 rows, never A2.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_FMT_E4M3 0 /* MXFP8 activations (A8W4)           */
#define ORACLE_FMT_E2M1 1 /* MXFP4 activations (A4W4) / weights */

/* ---------------------------------------------------------------------- */
/* Codebooks                                                               */
/* ---------------------------------------------------------------------- */

/* E2M1 (OCP MX FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Written out code by code. */
static const double E2M1_VALUE[16] = {
    0.0,  0.5,  1.0,  1.5,  2.0,  3.0,  4.0,  6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0};

/* E4M3 (OCP MX FP8, "fn" variant): 1 sign, 4 exponent bits (bias 7), 3
 * mantissa bits; exponent field 15 with mantissa 7 is NaN, there is no
 * infinity; largest finite magnitude 448.  Filled once from the definition. */
static double E4M3_VALUE[256];
/* E8M0 scale values 2^(s-127), s = 0..254 (255 is NaN). */
static double E8M0_VALUE[256];
static int e4m3_ready = 0;

static void e4m3_build(void) {
  for (int s = 0; s < 256; ++s) E8M0_VALUE[s] = (s == 255) ? NAN : ldexp(1.0, s - 127);
  for (int c = 0; c < 256; ++c) {
    int sign = (c >> 7) & 1;
    int ef = (c >> 3) & 15;
    int m = c & 7;
    double mag;
    if (ef == 15 && m == 7) {
      mag = NAN;
    } else if (ef == 0) {
      mag = ldexp((double)m / 8.0, -6); /* subnormal: 0.m * 2^(1-7) */
    } else {
      mag = ldexp(1.0 + (double)m / 8.0, ef - 7);
    }
    E4M3_VALUE[c] = sign ? -mag : mag;
  }
  e4m3_ready = 1;
}

double oracle_e2m1_decode(int code) { return E2M1_VALUE[code & 15]; }

double oracle_e4m3_decode(int code) {
  if (!e4m3_ready) e4m3_build();
  return E4M3_VALUE[code & 255];
}

/* E8M0: an unsigned biased exponent, value 2^(s-127); 0xFF is NaN. */
double oracle_e8m0_decode(int s) {
  if ((s & 255) == 255) return NAN;
  return ldexp(1.0, (s & 255) - 127);
}

static int fmt_emax(int fmt) { return fmt == ORACLE_FMT_E4M3 ? 8 : 2; }
static int fmt_ncodes(int fmt) { return fmt == ORACLE_FMT_E4M3 ? 256 : 16; }
static int fmt_signbit(int fmt) { return fmt == ORACLE_FMT_E4M3 ? 0x80 : 0x8; }
static double fmt_decode(int fmt, int c) {
  return fmt == ORACLE_FMT_E4M3 ? oracle_e4m3_decode(c) : oracle_e2m1_decode(c);
}

/* Encode an already-scaled value y to the nearest code of the format by a
 * plain search over every non-NaN, non-negative code; ties go to the code
 * whose least-significant bit is 0 (the even mantissa).  Magnitudes beyond
 * the largest finite value land on it (satfinite).  The sign bit is copied
 * from y, also when the magnitude rounds to zero. */
int oracle_mx_encode(double y, int fmt) {
  if (fmt == ORACLE_FMT_E4M3 && !e4m3_ready) e4m3_build();
  int neg = signbit(y) ? 1 : 0;
  double a = fabs(y);
  int sat = fmt == ORACLE_FMT_E4M3 ? 0x7E : 0x7; /* +448 / +6 */
  if (a >= fmt_decode(fmt, sat)) return neg ? (sat | fmt_signbit(fmt)) : sat; /* satfinite */
  int best = 0;
  double best_err = INFINITY;
  int half = fmt_ncodes(fmt) / 2; /* non-negative codes are 0 .. half-1 */
  for (int c = 0; c < half; ++c) {
    double v = fmt_decode(fmt, c);
    if (isnan(v)) continue;
    double err = fabs(v - a);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return neg ? (best | fmt_signbit(fmt)) : best;
}

/* Scale byte of one block from its largest magnitude (fp32). */
int oracle_mx_scale_byte(float amax, int fmt) {
  uint32_t bits;
  memcpy(&bits, &amax, 4);
  int ef = (int)((bits >> 23) & 0xFF);
  if (ef == 0) return 0; /* zero or subnormal block */
  int floor_log2 = ef - 127; /* exact for every normal fp32 */
  int s = floor_log2 - fmt_emax(fmt) + 127;
  if (s < 0) s = 0;
  if (s > 254) s = 254;
  return s;
}

/* Quantise one block of 32 fp32 values: writes 32 codes (one per byte) and
 * the scale byte. */
void oracle_mx_quantize_block(const float* v, int fmt, uint8_t* codes, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  int s = oracle_mx_scale_byte(amax, fmt);
  *scale = (uint8_t)s;
  uint32_t bits;
  memcpy(&bits, &amax, 4);
  int degenerate = ((bits >> 23) & 0xFF) == 0;
  double X = ldexp(1.0, s - 127);
  for (int i = 0; i < 32; ++i) {
    if (degenerate) {
      codes[i] = (uint8_t)(signbit(v[i]) ? fmt_signbit(fmt) : 0);
    } else {
      codes[i] = (uint8_t)oracle_mx_encode((double)v[i] / X, fmt);
    }
  }
}

/* ---------------------------------------------------------------------- */
/* Row quantisation (rows x K, K a multiple of 32)                          */
/* codes: E4M3 -> K bytes per row; E2M1 -> K/2 bytes per row, element 2i in */
/* the low nibble.  scales: row-major [rows, K/32].                         */
/* ---------------------------------------------------------------------- */

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint16_t f64_to_bf16_rne(double d) {
  /* Round to the nearest bf16, ties to even.  Done in two steps that are
   * each exact or correctly rounded: double -> fp32 would double-round, so
   * instead work from the double directly. */
  if (isnan(d)) return 0x7FC0;
  if (d == 0.0) return signbit(d) ? 0x8000 : 0x0000;
  int neg = d < 0;
  double a = fabs(d);
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
  int exp_unb = e - 1; /* a in [2^exp_unb, 2^(exp_unb+1)) */
  if (exp_unb < -126) exp_unb = -126; /* bf16 subnormal range */
  double q = ldexp(1.0, exp_unb - 7); /* spacing of bf16 values here */
  double r = a / q;
  double fl = floor(r);
  double frac = r - fl;
  double n;
  if (frac > 0.5) n = fl + 1.0;
  else if (frac < 0.5) n = fl;
  else n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double val = n * q;
  if (val >= ldexp(1.0, 128)) { /* overflow -> inf */
    return neg ? 0xFF80 : 0x7F80;
  }
  float f = (float)val; /* exact: val is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t h = (uint16_t)(u >> 16);
  return neg ? (uint16_t)(h | 0x8000) : h;
}

uint16_t oracle_f64_to_bf16(double d) { return f64_to_bf16_rne(d); }

static void quantize_row_f32(const float* v, int K, int fmt, uint8_t* codes_row, uint8_t* scales_row) {
  uint8_t c[32];
  for (int b = 0; b < K / 32; ++b) {
    oracle_mx_quantize_block(v + 32 * b, fmt, c, &scales_row[b]);
    for (int i = 0; i < 32; ++i) {
      int col = 32 * b + i;
      if (fmt == ORACLE_FMT_E4M3) {
        codes_row[col] = c[i];
      } else {
        uint8_t* byte = &codes_row[col / 2];
        if ((col & 1) == 0) *byte = (uint8_t)((*byte & 0xF0) | (c[i] & 0x0F));
        else *byte = (uint8_t)((*byte & 0x0F) | ((c[i] & 0x0F) << 4));
      }
    }
  }
}

static int64_t row_code_bytes(int K, int fmt) { return fmt == ORACLE_FMT_E4M3 ? K : K / 2; }

void oracle_quantize_rows_f32(const float* v, int64_t rows, int K, int fmt, uint8_t* codes, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r)
    quantize_row_f32(v + r * K, K, fmt, codes + r * row_code_bytes(K, fmt), scales + r * (K / 32));
}

void oracle_quantize_rows_bf16(const uint16_t* x, int64_t rows, int K, int fmt, uint8_t* codes, uint8_t* scales) {
  float* tmp = (float*)malloc(sizeof(float) * (size_t)K);
  for (int64_t r = 0; r < rows; ++r) {
    for (int i = 0; i < K; ++i) tmp[i] = bf16_to_f32(x[r * K + i]);
    quantize_row_f32(tmp, K, fmt, codes + r * row_code_bytes(K, fmt), scales + r * (K / 32));
  }
  free(tmp);
}

/* Decode one element (column col) of a quantised row to its real value. */
static double dequant_elem(const uint8_t* codes_row, const uint8_t* scales_row, int col, int fmt) {
  int code;
  if (fmt == ORACLE_FMT_E4M3) code = codes_row[col];
  else code = (col & 1) ? (codes_row[col / 2] >> 4) & 15 : codes_row[col / 2] & 15;
  return fmt_decode(fmt, code) * E8M0_VALUE[scales_row[col / 32]];
}

void oracle_dequantize_rows(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, int fmt, double* out) {
  if (!e4m3_ready) e4m3_build();
  for (int64_t r = 0; r < rows; ++r)
    for (int c = 0; c < K; ++c)
      out[r * K + c] = dequant_elem(codes + r * row_code_bytes(K, fmt), scales + r * (K / 32), c, fmt);
}

/* ---------------------------------------------------------------------- */
/* 1. Routing                                                              */
/* ---------------------------------------------------------------------- */

void oracle_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w) {
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    /* rank: repeatedly pick the largest remaining logit, lower index first */
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        int taken = 0;
        for (int i = 0; i < j; ++i) taken |= (ids[t * k + i] == e);
        if (taken) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: ties keep lower e */
      }
      ids[t * k + j] = best;
    }
    /* softmax over all E in double, then renormalise over the selected k */
    double m = -INFINITY;
    for (int e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp((double)l[e] - m);
    double sel = 0.0;
    double p[64];
    for (int j = 0; j < k; ++j) {
      p[j] = exp((double)l[ids[t * k + j]] - m) / z;
      sel += p[j];
    }
    for (int j = 0; j < k; ++j) w[t * k + j] = (float)(p[j] / sel);
  }
}

/* ---------------------------------------------------------------------- */
/* 2. Sort / permute                                                       */
/* sorted_pair[r] = q = t*k + j of the r-th row in (expert asc, q asc)     */
/* order; inv[q] = r; offsets has E+1 entries, offsets[E] = T*k.           */
/* ---------------------------------------------------------------------- */

void oracle_sort(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int64_t* offsets,
                 int32_t* sorted_pair, int32_t* inv) {
  int64_t R = T * (int64_t)k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t q = 0; q < R; ++q) counts[ids[q]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int64_t* next = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
  for (int e = 0; e < E; ++e) next[e] = offsets[e];
  for (int64_t q = 0; q < R; ++q) { /* visiting q in ascending order keeps it stable */
    int64_t r = next[ids[q]]++;
    sorted_pair[r] = (int32_t)q;
    inv[q] = (int32_t)r;
  }
  free(next);
}

/* ---------------------------------------------------------------------- */
/* 3-8. The expert layer for a list of tokens                              */
/* ---------------------------------------------------------------------- */

static float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

/*
 * x       bf16 [T, H]            logits fp32 [T, E]
 * w1      fp4  [E, 2I, H/2]      w1s    e8m0 [E, 2I, H/32]   (row 2j gate_j, 2j+1 up_j)
 * w2      fp4  [E, H, I/2]       w2s    e8m0 [E, H, I/32]
 * tokens  the n_tok token indices to evaluate (NULL: all T, in order)
 * out     bf16 [n_tok, H]
 * optional diagnostics (may be NULL), per evaluated token and slot:
 *   h_out   fp32 [n_tok, k, I]      a2_codes [n_tok, k, I or I/2]   a2_scales [n_tok, k, I/32]
 *   y2_out  fp32 [n_tok, k, H]
 * Returns 0, or -1 on bad arguments.
 */
#define ORACLE_OPT_H_BF16 1 /* round h to bf16 (nearest even) before its MX quantisation */
#define ORACLE_OPT_Y2_FP8 2 /* the weighted GEMM2 rows w_j * y2 (fp32 product) quantised to E4M3
                             with one E8M0 scale per 1x32 block, the combine summing their
                             dequantised values (FP8 transport of the stage-2 rows) */

static float round_bf16(float v) {
  const uint32_t bits = (uint32_t)f64_to_bf16_rne((double)v) << 16;
  float r;
  memcpy(&r, &bits, sizeof(r));
  return r;
}

int oracle_moe_forward_opts(const uint16_t* x, const float* logits, const uint8_t* w1, const uint8_t* w1s,
                            const uint8_t* w2, const uint8_t* w2s, int64_t T, int H, int I, int E, int k,
                            int act_fmt, const int64_t* tokens, int64_t n_tok, uint16_t* out, float* h_out,
                            uint8_t* a2_codes, uint8_t* a2_scales, float* y2_out, int nthreads, int opts) {
  if (H % 32 || I % 32 || k < 1 || k > 64 || k > E || T < 0) return -1;
  if (act_fmt != ORACLE_FMT_E4M3 && act_fmt != ORACLE_FMT_E2M1) return -1;
  if (!e4m3_ready) e4m3_build();
  if (tokens == NULL) n_tok = T;
  const int64_t w1_row = H / 2, w1s_row = H / 32, w2_row = I / 2, w2s_row = I / 32;
  const int64_t a2_row = row_code_bytes(I, act_fmt);
  if (nthreads < 1) nthreads = 1;

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int64_t it = 0; it < n_tok; ++it) {
    int64_t t = tokens ? tokens[it] : it;
    int32_t ids[64];
    float w[64];
    oracle_route(logits + t * E, 1, E, k, ids, w);

    /* 3. quantise this token's activation row */
    uint8_t* xq = (uint8_t*)malloc((size_t)row_code_bytes(H, act_fmt));
    uint8_t* xs = (uint8_t*)malloc((size_t)(H / 32));
    oracle_quantize_rows_bf16(x + t * H, 1, H, act_fmt, xq, xs);
    double* xd = (double*)malloc(sizeof(double) * (size_t)H);
    for (int c = 0; c < H; ++c) xd[c] = dequant_elem(xq, xs, c, act_fmt);

    double* acc = (double*)malloc(sizeof(double) * (size_t)H); /* combine accumulator */
    for (int n = 0; n < H; ++n) acc[n] = 0.0;
    float* h = (float*)malloc(sizeof(float) * (size_t)I);
    uint8_t* a2 = (uint8_t*)malloc((size_t)a2_row);
    uint8_t* a2s = (uint8_t*)malloc((size_t)(I / 32));
    double* a2d = (double*)malloc(sizeof(double) * (size_t)I);
    float* yw = (float*)malloc(sizeof(float) * (size_t)H); /* weighted row, FP8 transport */
    uint8_t* yq = (uint8_t*)malloc((size_t)H);
    uint8_t* ys = (uint8_t*)malloc((size_t)(H / 32));

    for (int j = 0; j < k; ++j) {
      int e = ids[j];
      /* 4-5. GEMM1 rows 2i (gate) and 2i+1 (up), then SwiGLU */
      for (int i = 0; i < I; ++i) {
        float g_up[2];
        for (int half = 0; half < 2; ++half) {
          int64_t n = 2 * (int64_t)i + half;
          const uint8_t* wr = w1 + ((int64_t)e * 2 * I + n) * w1_row;
          const uint8_t* ws = w1s + ((int64_t)e * 2 * I + n) * w1s_row;
          double s = 0.0;
          for (int c = 0; c < H; ++c) s += xd[c] * dequant_elem(wr, ws, c, ORACLE_FMT_E2M1);
          g_up[half] = (float)s;
        }
        h[i] = silu_mul(g_up[0], g_up[1]);
        if (opts & ORACLE_OPT_H_BF16) h[i] = round_bf16(h[i]);
      }
      /* 6. A2 */
      oracle_quantize_rows_f32(h, 1, I, act_fmt, a2, a2s);
      for (int c = 0; c < I; ++c) a2d[c] = dequant_elem(a2, a2s, c, act_fmt);
      /* 7-8. GEMM2 and the weighted combine */
      for (int n = 0; n < H; ++n) {
        const uint8_t* wr = w2 + ((int64_t)e * H + n) * w2_row;
        const uint8_t* ws = w2s + ((int64_t)e * H + n) * w2s_row;
        double s = 0.0;
        for (int c = 0; c < I; ++c) s += a2d[c] * dequant_elem(wr, ws, c, ORACLE_FMT_E2M1);
        float y = (float)s;
        if (y2_out) y2_out[(it * k + j) * (int64_t)H + n] = y;
        if (opts & ORACLE_OPT_Y2_FP8) yw[n] = w[j] * y;
        else acc[n] += (double)w[j] * (double)y;
      }
      if (opts & ORACLE_OPT_Y2_FP8) {
        oracle_quantize_rows_f32(yw, 1, H, ORACLE_FMT_E4M3, yq, ys);
        for (int n = 0; n < H; ++n) acc[n] += dequant_elem(yq, ys, n, ORACLE_FMT_E4M3);
      }
      if (h_out) memcpy(h_out + (it * k + j) * (int64_t)I, h, sizeof(float) * (size_t)I);
      if (a2_codes) memcpy(a2_codes + (it * k + j) * a2_row, a2, (size_t)a2_row);
      if (a2_scales) memcpy(a2_scales + (it * k + j) * (int64_t)(I / 32), a2s, (size_t)(I / 32));
    }
    for (int n = 0; n < H; ++n) out[it * (int64_t)H + n] = f64_to_bf16_rne(acc[n]);
    free(xq); free(xs); free(xd); free(acc); free(h); free(a2); free(a2s); free(a2d); free(yw); free(yq); free(ys);
  }
  return 0;
}

/* The layer as the method defines it (h quantised from fp32). */
int oracle_moe_forward(const uint16_t* x, const float* logits, const uint8_t* w1, const uint8_t* w1s,
                       const uint8_t* w2, const uint8_t* w2s, int64_t T, int H, int I, int E, int k,
                       int act_fmt, const int64_t* tokens, int64_t n_tok, uint16_t* out, float* h_out,
                       uint8_t* a2_codes, uint8_t* a2_scales, float* y2_out, int nthreads) {
  return oracle_moe_forward_opts(x, logits, w1, w1s, w2, w2s, T, H, I, E, k, act_fmt, tokens, n_tok, out, h_out,
                                 a2_codes, a2_scales, y2_out, nthreads, 0);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
