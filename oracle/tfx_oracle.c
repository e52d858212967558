/*
 * tfx_oracle.c -- plain CPU oracle for routed-expert MoE over MXFP4 weights.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The CUDA library never calls it, and the two share
 * no code, header, table or helper.
 *
 * What it computes, per token row r and routed slot j (expert e = ids[r][j]):
 *   g = x . Wg_e,  u = x . Wu_e,  h = silu(g) * u,  h quantised to the launch's activation
 *   format,  d = h . Wd_e,  y[r] = sum_j w[r][j] * d[r][j]  rounded to bf16.
 * Source: "dsv41 metal: decode experts decode an expert's weights once for all of its
 * rows" (TensorFold PR #2983), section "What this changes" and the commit message of the
 * rows kernels ("decode each 32-group of an expert's MXFP4 weights once per pass").
 *
 * Two evaluation modes:
 *   float64  -- the definition: every product and sum in double, naive loops. Each value
 *               also carries a "mass" (sum of |terms|, propagated through the stages) used
 *               by the tolerance |err| <= 1e-3 * mass + 1e-6.
 *   fp32 chain -- the evaluation order the pages fix for one row ("Why it is exact" in
 *               "What this changes"; the owner's review of ds_rows_chains): for each
 *               32-group, a sequential fma chain of the 32 unscaled products from zero in
 *               k order; then the group's scale applied by one fma into accumulator
 *               (group index mod 8); then the eight-way tree
 *               ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)).
 *
 * Element formats are written from their published definitions:
 *   OCP Microscaling Formats (MX) v1.0: FP4 E2M1 elements (bias 1, values +-{0, .5, 1,
 *   1.5, 2, 3, 4, 6}), E8M0 block scales (2^(e-127), 0xFF = NaN), 32 elements a block.
 *   OCP 8-bit Floating Point (OFP8): E4M3 (bias 7, no infinities, S.1111.111 = NaN,
 *   max 448). bf16: IEEE-754 binary32 with the low 16 bits dropped, rounded to nearest even.
 *
 * Compile with -ffp-contract=off so that every fp32 operation rounds where written.
 *
 * Planted controls: built with -DTFXO_CTL=n (n > 0), one deliberate mistake of a known kind
 * is compiled in (the nibble order, the tree, the scale index, one accumulator for every
 * group, the weight scale's bias, the chain's k order, the combine's slot order, the E4M3
 * tie rule, the mass as |sum| instead of sum of |terms|, the SwiGLU mass without its
 * g (1 - s) derivative term, the combine mass with signed weights, bf16 rounding of a
 * float64 through binary32), so that a test can show
 * that the pins catch it. TFXO_CTL 0, the default, is the oracle as it ships.
 */
#ifndef TFXO_CTL
#define TFXO_CTL 0
#endif

#include <math.h>
#include <stdint.h>
#include <string.h>

#include "tfx_oracle.h"

/* ------------------------------------------------------------------ element formats */

/* OCP MX v1.0, FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. */
double tfxo_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double v = (e == 0) ? (m * 0.5) : ldexp(1.0 + m * 0.5, e - 1);
  return s ? -v : v;
}

/* OCP OFP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN. */
double tfxo_e4m3_value(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* OCP MX v1.0 E8M0 scale: 2^(e-127); 0xFF is NaN. */
double tfxo_ue8m0_value(int code) {
  if ((code & 255) == 255) return NAN;
  return ldexp(1.0, (code & 255) - 127);
}

static float ue8m0_f32(int code) {
  if ((code & 255) == 255) return NAN;
  return ldexpf(1.0f, (code & 255) - 127); /* exact, including the subnormal 2^-127 */
}

float tfxo_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* IEEE round-to-nearest-even from binary32 to bf16; NaN stays NaN (made quiet). */
uint16_t tfxo_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* IEEE round-to-nearest-even from binary64 straight to bf16, one rounding (no binary32 step in
 * between, which could round a value just past a bf16 midpoint onto it and then to even); values
 * at or beyond the midpoint above the largest finite bf16 become infinity; NaN -> quiet NaN. */
uint16_t tfxo_f64_to_bf16(double v) {
  if (isnan(v)) return signbit(v) ? 0xFFC0u : 0x7FC0u;
  uint16_t s = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (a == 0.0) return s;
  if (isinf(a)) return s | 0x7F80u;
#if TFXO_CTL == 12
  return tfxo_f32_to_bf16((float)v); /* planted: rounded to binary32 first, then to bf16 */
#else
  int ex;
  frexp(a, &ex);
  ex -= 1;                              /* a in [2^ex, 2^(ex+1)) */
  int q = (ex < -126) ? -133 : ex - 7;  /* spacing of the bf16 grid around a (8 significant bits) */
  double val = ldexp(rint(ldexp(a, -q)), q);
  if (val >= ldexp(1.0, 128)) return s | 0x7F80u;
  float f = (float)val;                 /* exact: val lies on the bf16 grid */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(s | ((u >> 16) & 0x7FFFu));
#endif
}

/* Nearest E4M3 code to v, ties to even, magnitudes beyond 448 saturated to 448; NaN -> 0x7F. */
int tfxo_e4m3_encode(double v) {
  if (isnan(v)) return 0x7F;
  int s = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  if (a >= 448.0) return s | 0x7E;
  if (a == 0.0) return s;
  int ex;
  frexp(a, &ex);
  ex -= 1;                              /* a in [2^ex, 2^(ex+1)) */
  int q = (ex < -6) ? -9 : ex - 3;      /* spacing of the E4M3 grid around a */
#if TFXO_CTL == 8
  double r = round(ldexp(a, -q));       /* planted: ties away from zero */
#else
  double r = rint(ldexp(a, -q));        /* default rounding mode: nearest, ties to even */
#endif
  double val = ldexp(r, q);
  if (val >= 448.0) return s | 0x7E;
  if (val < ldexp(1.0, -6)) return s | (int)(val * 512.0); /* subnormals: m * 2^-9 */
  int ev;
  frexp(val, &ev);
  ev -= 1;
  int m3 = (int)((ldexp(val, -ev) - 1.0) * 8.0);
  return s | ((ev + 7) << 3) | m3;
}

/* ------------------------------------------------------------------ activation quantiser
 * A block of 32 values becomes 32 E4M3 codes plus one E8M0 scale (OCP MX v1.0 rule:
 * shared exponent floor(log2(amax)) - 8, where 8 is the largest E4M3 exponent; elements
 * divided by the scale, rounded to nearest even and saturated to +-448). amax 0 gives
 * scale code 127; a NaN or infinity in the block gives scale code 0xFF (and NaN elements).
 */
static void quant_block(const double* v, uint8_t* codes, uint8_t* scale) {
  double amax = 0.0;
  int bad = 0;
  for (int i = 0; i < 32; i++) {
    if (isnan(v[i]) || isinf(v[i])) bad = 1;
    else if (fabs(v[i]) > amax) amax = fabs(v[i]);
  }
  if (bad) {
    *scale = 0xFF;
    for (int i = 0; i < 32; i++) codes[i] = 0x7F;
    return;
  }
  int sc = 127;
  if (amax > 0.0) {
    int e2;
    frexp(amax, &e2);                   /* amax in [2^(e2-1), 2^e2) */
    int x = (e2 - 1) - 8;
    sc = x + 127;
    if (sc < 0) sc = 0;
    if (sc > 254) sc = 254;
  }
  *scale = (uint8_t)sc;
  for (int i = 0; i < 32; i++) codes[i] = (uint8_t)tfxo_e4m3_encode(ldexp(v[i], 127 - sc));
}

void tfxo_quant_e4m3_f32(int n, const float* h, uint8_t* codes, uint8_t* scales) {
  double tmp[32];
  for (int b = 0; b < n / 32; b++) {
    for (int i = 0; i < 32; i++) tmp[i] = (double)h[32 * b + i];
    quant_block(tmp, codes + 32 * b, scales + b);
  }
}

void tfxo_quant_e4m3_f64(int n, const double* h, uint8_t* codes, uint8_t* scales) {
  for (int b = 0; b < n / 32; b++) quant_block(h + 32 * b, codes + 32 * b, scales + b);
}

void tfxo_round_bf16(int n, const float* h, uint16_t* out) {
  for (int i = 0; i < n; i++) out[i] = tfxo_f32_to_bf16(h[i]);
}

void tfxo_round_bf16_f64(int n, const double* h, uint16_t* out) {
  for (int i = 0; i < n; i++) out[i] = tfxo_f64_to_bf16(h[i]);
}

/* ------------------------------------------------------------------ routing
 * Expert-major row lists ("every expert's rows"): for each expert, the (row, slot) pairs
 * routed to it in ascending (row, slot) order; the active experts in ascending id.
 * An id outside [0, E) sets TFXO_ST_RANGE; an id equal to an earlier slot's id in the same
 * row sets TFXO_ST_DUP. Either pair is left out of every list.
 */
int tfxo_route(const int32_t* ids, int R, int k, int E, int32_t* offs, int32_t* pair_row,
               int32_t* pair_slot, int32_t* active, int32_t* n_active) {
  int status = 0;
  for (int e = 0; e <= E; e++) offs[e] = 0;
  for (int r = 0; r < R; r++)
    for (int j = 0; j < k; j++) {
      int e = ids[r * k + j];
      if (e < 0 || e >= E) { status |= TFXO_ST_RANGE; continue; }
      int dup = 0;
      for (int jj = 0; jj < j; jj++) if (ids[r * k + jj] == e) dup = 1;
      if (dup) { status |= TFXO_ST_DUP; continue; }
      offs[e + 1]++;
    }
  for (int e = 0; e < E; e++) offs[e + 1] += offs[e];
  int na = 0;
  for (int e = 0; e < E; e++) {
    int pos = offs[e];
    for (int r = 0; r < R; r++)
      for (int j = 0; j < k; j++) {
        if (ids[r * k + j] != e) continue;
        int dup = 0;
        for (int jj = 0; jj < j; jj++) if (ids[r * k + jj] == e) dup = 1;
        if (dup) continue;
        pair_row[pos] = r;
        pair_slot[pos] = j;
        pos++;
      }
    if (offs[e + 1] > offs[e]) active[na++] = e;
  }
  *n_active = na;
  return status;
}

/* ------------------------------------------------------------------ one output, two modes */

static int nibble(const uint8_t* codes, int k) {
  uint8_t b = codes[k >> 1];
#if TFXO_CTL == 1
  return (k & 1) ? (b & 15) : (b >> 4); /* planted: nibble order swapped */
#else
  return (k & 1) ? (b >> 4) : (b & 15); /* the lower k sits in the low nibble */
#endif
}

/* Unscaled element values of one activation row, and the fp32 value of each group's scale. */
static void act_row_f32(int kind, int K, const void* x, const uint8_t* sx, float* xc, float* xs) {
  if (kind == TFXO_ACT_E4M3) {
    const uint8_t* c = (const uint8_t*)x;
    for (int i = 0; i < K; i++) xc[i] = (float)tfxo_e4m3_value(c[i]);
    for (int g = 0; g < K / 32; g++) xs[g] = ue8m0_f32(sx[g]);
  } else {
    const uint16_t* b = (const uint16_t*)x;
    for (int i = 0; i < K; i++) xc[i] = tfxo_bf16_to_f32(b[i]);
    for (int g = 0; g < K / 32; g++) xs[g] = 1.0f;
  }
}

static void act_row_f64(int kind, int K, const void* x, const uint8_t* sx, double* xh) {
  if (kind == TFXO_ACT_E4M3) {
    const uint8_t* c = (const uint8_t*)x;
    for (int i = 0; i < K; i++) xh[i] = tfxo_e4m3_value(c[i]) * tfxo_ue8m0_value(sx[i / 32]);
  } else {
    const uint16_t* b = (const uint16_t*)x;
    for (int i = 0; i < K; i++) xh[i] = (double)tfxo_bf16_to_f32(b[i]);
  }
}

/* fp32 chain for one output: weight row (codes [K/2], scales [K/32]) against one activation row. */
float tfxo_chain_dot(int K, const uint8_t* wc, const uint8_t* ws, const float* xc, const float* xs) {
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int g = 0; g < K / 32; g++) {
    float p = 0.0f;
#if TFXO_CTL == 6
    for (int t = 31; t >= 0; t--) { /* planted: the chain runs from the last k down */
      int k = 32 * g + t;
      p = fmaf((float)tfxo_e2m1_value(nibble(wc, k)), xc[k], p);
    }
#else
    for (int t = 0; t < 32; t++) {
      int k = 32 * g + t;
      p = fmaf((float)tfxo_e2m1_value(nibble(wc, k)), xc[k], p);
    }
#endif
#if TFXO_CTL == 3
    float s = ue8m0_f32(ws[0]) * xs[0]; /* planted: the first group's scale for the whole row */
#elif TFXO_CTL == 5
    float s = ldexpf(1.0f, (int)ws[g] - 128) * xs[g]; /* planted: E8M0 bias off by one */
#else
    float s = ue8m0_f32(ws[g]) * xs[g];
#endif
#if TFXO_CTL == 4
    acc[0] = fmaf(p, s, acc[0]); /* planted: every group into one accumulator */
#else
    acc[g & 7] = fmaf(p, s, acc[g & 7]);
#endif
  }
#if TFXO_CTL == 2
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7])); /* planted: tree */
#else
  return ((acc[0] + acc[4]) + (acc[2] + acc[6])) + ((acc[1] + acc[5]) + (acc[3] + acc[7]));
#endif
}

/* float64 definition for one output, with its mass. */
double tfxo_f64_dot(int K, const uint8_t* wc, const uint8_t* ws, const double* xh, double* mass) {
  double s = 0.0, m = 0.0;
  for (int k = 0; k < K; k++) {
    double w = tfxo_e2m1_value(nibble(wc, k)) * tfxo_ue8m0_value(ws[k / 32]);
    double t = w * xh[k];
    s += t;
    m += fabs(t);
  }
#if TFXO_CTL == 9
  m = fabs(s); /* planted: the mass taken as |sum of terms| instead of the sum of |terms| */
#endif
  *mass = m;
  return s;
}

/* ------------------------------------------------------------------ stages, one (expert, row) pair
 * Canonical layouts of one expert: Wg, Wu codes [I][H/2], scales [I][H/32];
 * Wd codes [H][I/2], scales [H][I/32].  Activations: E4M3 codes [K] + E8M0 scales [K/32],
 * or bf16 [K].
 */
void tfxo_gateup_chain(int H, int I, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                       const uint8_t* su, int kind, const void* x, const uint8_t* sx, float* xbuf,
                       float* g, float* u) {
  float* xc = xbuf;
  float* xs = xbuf + H;
  act_row_f32(kind, H, x, sx, xc, xs);
  for (int n = 0; n < I; n++) {
    g[n] = tfxo_chain_dot(H, wg + (size_t)n * (H / 2), sg + (size_t)n * (H / 32), xc, xs);
    u[n] = tfxo_chain_dot(H, wu + (size_t)n * (H / 2), su + (size_t)n * (H / 32), xc, xs);
  }
}

void tfxo_gateup_f64(int H, int I, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu,
                     const uint8_t* su, int kind, const void* x, const uint8_t* sx, double* xbuf,
                     double* g, double* u, double* mg, double* mu) {
  act_row_f64(kind, H, x, sx, xbuf);
  for (int n = 0; n < I; n++) {
    g[n] = tfxo_f64_dot(H, wg + (size_t)n * (H / 2), sg + (size_t)n * (H / 32), xbuf, &mg[n]);
    u[n] = tfxo_f64_dot(H, wu + (size_t)n * (H / 2), su + (size_t)n * (H / 32), xbuf, &mu[n]);
  }
}

/* SwiGLU epilogue in fp32: h = (g / (1 + exp(-g))) * u, each operation rounded. */
void tfxo_silu_mul_f32(int n, const float* g, const float* u, float* h) {
  for (int i = 0; i < n; i++) {
    float e = expf(-g[i]);
    float den = 1.0f + e;
    float sg = g[i] / den;
    h[i] = sg * u[i];
  }
}

/* The same in float64, with the first-order propagated mass:
 * mass_h = |silu'(g)| mass_g |u| + |silu(g)| mass_u + |h|, silu'(g) = s (1 + g (1 - s)). */
void tfxo_silu_mul_f64(int n, const double* g, const double* u, const double* mg, const double* mu,
                       double* h, double* mh) {
  for (int i = 0; i < n; i++) {
    double s = 1.0 / (1.0 + exp(-g[i]));
    double si = g[i] * s;
#if TFXO_CTL == 10
    double d = s; /* planted: silu'(g) taken as the sigmoid alone, the g (1 - s) term dropped */
#else
    double d = s * (1.0 + g[i] * (1.0 - s));
#endif
    h[i] = si * u[i];
    mh[i] = fabs(d) * mg[i] * fabs(u[i]) + fabs(si) * mu[i] + fabs(h[i]);
  }
}

void tfxo_down_chain(int H, int I, const uint8_t* wd, const uint8_t* sd, int kind, const void* h,
                     const uint8_t* sh, float* xbuf, float* d) {
  float* hc = xbuf;
  float* hs = xbuf + I;
  act_row_f32(kind, I, h, sh, hc, hs);
  for (int m = 0; m < H; m++)
    d[m] = tfxo_chain_dot(I, wd + (size_t)m * (I / 2), sd + (size_t)m * (I / 32), hc, hs);
}

void tfxo_down_f64(int H, int I, const uint8_t* wd, const uint8_t* sd, int kind, const void* h,
                   const uint8_t* sh, double* xbuf, double* d, double* md) {
  act_row_f64(kind, I, h, sh, xbuf);
  for (int m = 0; m < H; m++)
    d[m] = tfxo_f64_dot(I, wd + (size_t)m * (I / 2), sd + (size_t)m * (I / 32), xbuf, &md[m]);
}

/* Combine one row: y = fma chain over the slots in slot order from +0, then bf16 (RNE). */
void tfxo_combine_chain(int k, int H, const float* d /*[k][H]*/, const float* w /*[k]*/,
                        uint16_t* y_bf16, float* y_f32) {
  for (int m = 0; m < H; m++) {
    float y = 0.0f;
#if TFXO_CTL == 7
    for (int j = k - 1; j >= 0; j--) y = fmaf(w[j], d[(size_t)j * H + m], y); /* planted: slots reversed */
#else
    for (int j = 0; j < k; j++) y = fmaf(w[j], d[(size_t)j * H + m], y);
#endif
    if (y_f32) y_f32[m] = y;
    y_bf16[m] = tfxo_f32_to_bf16(y);
  }
}

void tfxo_combine_f64(int k, int H, const double* d, const double* md, const float* w, double* y,
                      double* my) {
  for (int m = 0; m < H; m++) {
    double s = 0.0, ms = 0.0;
    for (int j = 0; j < k; j++) {
      s += (double)w[j] * d[(size_t)j * H + m];
#if TFXO_CTL == 11
      ms += (double)w[j] * md[(size_t)j * H + m]; /* planted: the weight's sign kept in the mass */
#else
      ms += fabs((double)w[j]) * md[(size_t)j * H + m];
#endif
    }
    y[m] = s;
    my[m] = ms;
  }
}
