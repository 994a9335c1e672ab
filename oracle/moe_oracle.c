/*
 * moe_oracle.c -- plain fp64 CPU oracle for the dropless mixture-of-experts
 * expert layer (router softmax + top-k, dispatch, SwiGLU experts, weighted
 * combine; and the backward of all of it).
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code with the CUDA
 * library: no headers, no helpers, no tables.  Inputs come from the seeded
 * generators; every expected value the tests use comes from here.
 *
 * Definition followed (the method reaches the plain dropless MoE result):
 *   - A learned router picks the Top-K experts for every token ("NVIDIA lleva
 *     el MoE de DeepSeek-V3 de 103 a 1.068 TFLOPS", intro).  Softmax over all
 *     E logits, keep the k largest, renormalise the kept probabilities.
 *   - Dropless: every token is processed by every expert it chose, however
 *     unbalanced the loads ("En que se diferencia el MoE sin descartes...").
 *   - Dispatch permutes tokens into per-expert groups; the grouped MLP runs
 *     two GEMMs per expert with SwiGLU between them; combine restores token
 *     order and accumulates the per-expert results ("Figura 3", "Optimizacion
 *     2"; the Mega MoE description in the aisight.pl and diariobitcoin.com
 *     write-ups names the two expert linears, SwiGLU and combine).
 * Readings where the pages are silent (each listed in the design notes):
 *   - top-k ranks by fp32 logit, larger first; equal logits -> lower expert
 *     index first.  Softmax is monotone, so this is the top-k of the
 *     probabilities without rounding ties.
 *   - SwiGLU(g, u) = silu(g) * u with g = x.W_gate, u = x.W_up, no biases.
 *   - rows inside an expert group are in ascending token order.
 *   - d(router weight) is returned as the gradient with respect to the logits.
 *   - fp8_bwd: each backward GEMM operand is quantised to MXFP8 (E4M3 values,
 *     one power-of-two UE8M0 scale per 32 consecutive elements along the GEMM's
 *     reduction dimension); blocks along tokens start at each expert's first row.
 *     The router weight is not folded into a quantised operand: dA's operands
 *     are dy (along H) and W_down, with w applied to the product in full
 *     precision; dW_down's operands are w*a and dy (along tokens).
 *     Every code is decided on the bf16 tensors the backward holds: the forward
 *     runs in BF16, so the activations it saves (g, u) are bf16 when dSwiGLU
 *     reads them, and dg, du and w*a are rounded to bf16 (nearest-even) before
 *     they are quantised.  Where floating point decides an integer code, both
 *     this oracle and the GPU take the decision on the same bf16 values.
 *   - mxfp8 (the forward GEMMs in MXFP8 as well): x along H and W_gate/W_up
 *     along H (their reduction dimension) for GEMM1; a = silu(g) u, rounded to
 *     bf16 (the forward's bf16 tensor), and W_down along I for GEMM2.  g and u
 *     are the products of the dequantised operands (not rounded: the backward
 *     reads them as bf16 through the fp8_bwd rule above); the backward of this
 *     mode is the fp8_bwd backward on these forward values.
 *
 * Arithmetic: fp64 throughout; bf16 inputs are widened exactly.  The oracle
 * never rounds intermediates.  Loops run in a fixed order; OpenMP only splits
 * independent tokens or experts, so results do not depend on thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

typedef struct {
  int64_t T;
  int32_t H, I, E, k;
} oracle_shape;

static double bf(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Nearest bf16 (8 significant bits, fp32's exponent range), ties to even;
 * magnitudes that round past the largest finite bf16 become infinite. */
EXPORT double oracle_round_bf16(double v) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  double a = fabs(v), r;
  if (a < 0x1p-126) {
    r = nearbyint(a / 0x1p-133) * 0x1p-133; /* subnormal spacing 2^-133 */
  } else {
    int ex;
    double f = frexp(a, &ex);                 /* a = f 2^ex, f in [0.5, 1) */
    r = ldexp(nearbyint(ldexp(f, 8)), ex - 8); /* 8 significant bits */
    if (r > 0x1.FEp127) r = INFINITY;
  }
  return v < 0 ? -r : r;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
static double silu(double z) { return z * sigmoid(z); }

/* ------------------------------------------------------------------------- */
/* MXFP8 (OCP Microscaling v1.0 element format E4M3, scale format E8M0).      */
/* ------------------------------------------------------------------------- */

/* E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities; the only
 * NaN pattern is S.1111.111, so the largest finite magnitude is 1.75*2^8 = 448.
 * Subnormals (exponent field 0) are m * 2^-9.  Round to nearest, ties to even;
 * magnitudes beyond 448 saturate to 448. */
EXPORT uint8_t oracle_e4m3_encode(double v) {
  uint8_t s = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (isnan(v)) return 0x7F;
  if (a >= 0x1p-6) {
    int ex;
    double f = frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;            /* a = q * 2^e, q in [1, 2) */
    double q = f * 2.0;
    double m = nearbyint((q - 1.0) * 8.0); /* 0..8, ties to even */
    if (m == 8.0) {
      m = 0.0;
      e += 1;
    }
    if (e > 8 || (e == 8 && m == 7.0)) return (uint8_t)(s | 0x7E); /* saturate: 448 */
    return (uint8_t)(s | ((e + 7) << 3) | (int)m);
  }
  double m = nearbyint(a / 0x1p-9); /* 0..8 */
  if (m == 8.0) return (uint8_t)(s | 0x08); /* rounds up to the smallest normal */
  return (uint8_t)(s | (int)m);
}

EXPORT double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Shared scale of one block: the smallest power of two 2^X such that
 * amax / 2^X <= 448, so that no element of the block saturates.  X is clamped
 * to the E8M0 range [-127, 127]; an all-zero block takes X = -127.
 * Returns X; the E8M0 code is X + 127. */
EXPORT int oracle_mx_scale_exp(double amax) {
  if (!(amax > 0.0)) return -127;
  int X = ilogb(amax) - 8;
  if (amax > ldexp(448.0, X)) X += 1;
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  return X;
}

/* Quantise n (<= 32) values read with the given stride: out (dequantised
 * values, may be NULL), codes (may be NULL), returns the scale exponent. */
static int mx_block(const double *v, int n, int64_t stride, double *out, int64_t ostride,
                    uint8_t *codes) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) {
    double a = fabs(v[i * stride]);
    if (a > amax) amax = a;
  }
  int X = oracle_mx_scale_exp(amax);
  for (int i = 0; i < n; ++i) {
    uint8_t c = oracle_e4m3_encode(ldexp(v[i * stride], -X));
    if (codes) codes[i] = c;
    if (out) out[i * ostride] = ldexp(oracle_e4m3_decode(c), X);
  }
  return X;
}

/* Quantise-dequantise a vector of length len in blocks of 32 from its start. */
static void mx_vec(double *v, int64_t len, int64_t stride) {
  for (int64_t b = 0; b < len; b += 32) {
    int n = (int)((len - b) < 32 ? (len - b) : 32);
    mx_block(v + b * stride, n, stride, v + b * stride, stride, NULL);
  }
}

/* Rows of bf16 values quantised along the row in blocks of 32: codes [rows,len],
 * scale codes [rows, len/32] (E8M0 = X + 127), dequantised values as float
 * (exact: an E4M3 value times a power of two fits in fp32 here). */
EXPORT int oracle_mx_quantize_rows_bf16(int64_t rows, int64_t len, const uint16_t *in,
                                        uint8_t *codes, uint8_t *scales, float *deq) {
  if (len % 32) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double buf[32], o[32];
    uint8_t c[32];
    for (int64_t b = 0; b < len; b += 32) {
      for (int i = 0; i < 32; ++i) buf[i] = bf(in[r * len + b + i]);
      int X = mx_block(buf, 32, 1, o, 1, c);
      if (scales) scales[r * (len / 32) + b / 32] = (uint8_t)(X + 127);
      for (int i = 0; i < 32; ++i) {
        if (codes) codes[r * len + b + i] = c[i];
        if (deq) deq[r * len + b + i] = (float)o[i];
      }
    }
  }
  return 0;
}

/* Column-wise quantisation of bf16 rows [seg, seg+n) of a [rows, cols] matrix,
 * blocks of 32 rows starting at seg (the expert's first row); a partial last
 * block is padded with zeros.  codes [n_pad, cols], scales [n_pad/32, cols]. */
EXPORT int oracle_mx_quantize_cols_bf16(int64_t cols, int64_t seg, int64_t n, const uint16_t *in,
                                        uint8_t *codes, uint8_t *scales) {
  int64_t nb = (n + 31) / 32;
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < cols; ++c) {
    double buf[32];
    uint8_t cd[32];
    for (int64_t b = 0; b < nb; ++b) {
      for (int i = 0; i < 32; ++i) {
        int64_t r = b * 32 + i;
        buf[i] = r < n ? bf(in[(seg + r) * cols + c]) : 0.0;
      }
      int X = mx_block(buf, 32, 1, NULL, 1, cd);
      scales[b * cols + c] = (uint8_t)(X + 127);
      for (int i = 0; i < 32; ++i) codes[(b * 32 + i) * cols + c] = cd[i];
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Router: softmax over E, keep top-k, renormalise.                           */
/* ------------------------------------------------------------------------- */

/* Ranks expert a ahead of expert b for a token. */
static int ahead(float la, int a, float lb, int b) { return la > lb || (la == lb && a < b); }

static void route_token(int32_t E, int32_t k, const float *l, int32_t *idx, double *w, double *p) {
  /* probabilities */
  double mx = -INFINITY;
  for (int e = 0; e < E; ++e)
    if (l[e] > mx) mx = l[e];
  double z = 0.0;
  for (int e = 0; e < E; ++e) {
    p[e] = exp((double)l[e] - mx);
    z += p[e];
  }
  for (int e = 0; e < E; ++e) p[e] /= z;
  /* selection: k passes, each takes the best expert not yet taken */
  char taken[4096];
  memset(taken, 0, (size_t)E);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && (best < 0 || ahead(l[e], e, l[best], best))) best = e;
    taken[best] = 1;
    idx[j] = best;
  }
  /* renormalise over the kept set */
  double s = 0.0;
  for (int j = 0; j < k; ++j) s += p[idx[j]];
  for (int j = 0; j < k; ++j) w[j] = p[idx[j]] / s;
}

EXPORT int oracle_route(int64_t T, int32_t E, int32_t k, const float *logits, int32_t *topk_idx,
                        double *topk_w) {
  if (E < 1 || E > 4096 || k < 1 || k > E) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    double p[4096];
    route_token(E, k, logits + t * E, topk_idx + t * k, topk_w + t * k, p);
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Dispatch: per-expert counts, exclusive offsets, stable (token-ascending)    */
/* placement of every (token, choice) slot.                                   */
/* ------------------------------------------------------------------------- */

EXPORT int oracle_dispatch(int64_t T, int32_t E, int32_t k, const int32_t *topk_idx,
                           int32_t *counts, int32_t *offsets, int32_t *row_of_slot,
                           int32_t *slot_of_row) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t s = 0; s < T * k; ++s) {
    int e = topk_idx[s];
    if (e < 0 || e >= E) return -1;
    counts[e]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[t * k + j];
      int32_t row = offsets[e] + fill[e]++;
      row_of_slot[t * k + j] = row;
      slot_of_row[row] = (int32_t)(t * k + j);
    }
  free(fill);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* One expert on one token: g = x W_gate, u = x W_up, a = silu(g) u, y = a W_down */
/* ------------------------------------------------------------------------- */

typedef struct {
  const oracle_shape *sh;
  const uint16_t *x, *Wg, *Wu, *Wd, *dy;
  /* fp8_bwd: dequantised weights (quantised along each backward GEMM's K):
   * Wd along H, Wg/Wu along I.  NULL when not quantising. */
  const float *qWg, *qWu, *qWd;
  /* mxfp8 forward: dequantised weights quantised along each forward GEMM's K:
   * Wg/Wu along H, Wd along I.  NULL for the exact forward. */
  const float *fWg, *fWu, *fWd;
} ctx_t;

static void expert_fwd_mx(const ctx_t *c, int64_t t, int e, double *g, double *u, double *a,
                          double *y);

static void expert_fwd(const ctx_t *c, int64_t t, int e, double *g, double *u, double *a, double *y) {
  if (c->fWg) {
    expert_fwd_mx(c, t, e, g, u, a, y);
    return;
  }
  const int H = c->sh->H, I = c->sh->I;
  const uint16_t *xt = c->x + t * H;
  const uint16_t *wg = c->Wg + (int64_t)e * H * I, *wu = c->Wu + (int64_t)e * H * I;
  const uint16_t *wd = c->Wd + (int64_t)e * I * H;
  for (int i = 0; i < I; ++i) g[i] = u[i] = 0.0;
  for (int h = 0; h < H; ++h) {
    double xv = bf(xt[h]);
    for (int i = 0; i < I; ++i) {
      g[i] += xv * bf(wg[(int64_t)h * I + i]);
      u[i] += xv * bf(wu[(int64_t)h * I + i]);
    }
  }
  for (int i = 0; i < I; ++i) a[i] = silu(g[i]) * u[i];
  if (y) {
    for (int h = 0; h < H; ++h) y[h] = 0.0;
    for (int i = 0; i < I; ++i)
      for (int h = 0; h < H; ++h) y[h] += a[i] * bf(wd[(int64_t)i * H + h]);
  }
}

/* The same expert with its forward GEMMs in MXFP8: g = Q(x_t) . Q(W_gate[e])
 * (x along H, W along H), u likewise; a = silu(g) u; y = Q(bf16(a)) . Q(W_down[e])
 * (both along I). */
static void expert_fwd_mx(const ctx_t *c, int64_t t, int e, double *g, double *u, double *a,
                          double *y) {
  const int H = c->sh->H, I = c->sh->I;
  double *xq = malloc(sizeof(double) * (size_t)(H + I));
  double *aq = xq + H;
  for (int h = 0; h < H; ++h) xq[h] = bf(c->x[t * H + h]);
  mx_vec(xq, H, 1);
  const float *wg = c->fWg + (int64_t)e * H * I, *wu = c->fWu + (int64_t)e * H * I;
  for (int i = 0; i < I; ++i) g[i] = u[i] = 0.0;
  for (int h = 0; h < H; ++h)
    for (int i = 0; i < I; ++i) {
      g[i] += xq[h] * (double)wg[(int64_t)h * I + i];
      u[i] += xq[h] * (double)wu[(int64_t)h * I + i];
    }
  for (int i = 0; i < I; ++i) a[i] = silu(g[i]) * u[i];
  if (y) {
    const float *wd = c->fWd + (int64_t)e * I * H;
    for (int i = 0; i < I; ++i) aq[i] = oracle_round_bf16(a[i]);
    mx_vec(aq, I, 1);
    for (int h = 0; h < H; ++h) y[h] = 0.0;
    for (int i = 0; i < I; ++i)
      for (int h = 0; h < H; ++h) y[h] += aq[i] * (double)wd[(int64_t)i * H + h];
  }
  free(xq);
}

static void ctx_init(ctx_t *c, const oracle_shape *sh, const uint16_t *x, const uint16_t *Wg,
                     const uint16_t *Wu, const uint16_t *Wd, const uint16_t *dy, const float *qWg,
                     const float *qWu, const float *qWd) {
  c->sh = sh;
  c->x = x;
  c->Wg = Wg;
  c->Wu = Wu;
  c->Wd = Wd;
  c->dy = dy;
  c->qWg = qWg;
  c->qWu = qWu;
  c->qWd = qWd;
  c->fWg = c->fWu = c->fWd = NULL;
}

/* Forward-quantised weights (mxfp8): all three or none. */
static int ctx_forward_quant(ctx_t *c, const float *fWg, const float *fWu, const float *fWd) {
  if (!fWg && !fWu && !fWd) return 0;
  if (!fWg || !fWu || !fWd || c->sh->H % 32 || c->sh->I % 32) return -1;
  c->fWg = fWg;
  c->fWu = fWu;
  c->fWd = fWd;
  return 0;
}

/* Forward for a list of tokens: out[n] = sum_j w_j * y(t, S_j).  Optionally the
 * per-choice expert outputs y [n, k, H].  fWg/fWu/fWd: forward-quantised
 * weights (mxfp8) or NULL. */
EXPORT int oracle_forward(const oracle_shape *sh, const uint16_t *x, const int32_t *topk_idx,
                          const double *topk_w, const uint16_t *Wg, const uint16_t *Wu,
                          const uint16_t *Wd, const float *fWg, const float *fWu, const float *fWd,
                          int64_t ntok, const int64_t *tokens, double *out, double *y_all) {
  const int H = sh->H, I = sh->I, k = sh->k;
  ctx_t c;
  ctx_init(&c, sh, x, Wg, Wu, Wd, NULL, NULL, NULL, NULL);
  if (ctx_forward_quant(&c, fWg, fWu, fWd)) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t n = 0; n < ntok; ++n) {
    int64_t t = tokens[n];
    if (t < 0 || t >= sh->T) {
      bad = 1;
      continue;
    }
    double *g = malloc(sizeof(double) * (size_t)(3 * I + H));
    double *u = g + I, *a = u + I, *y = a + I;
    for (int h = 0; h < H; ++h) out[n * H + h] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[t * k + j];
      expert_fwd(&c, t, e, g, u, a, y);
      for (int h = 0; h < H; ++h) out[n * H + h] += topk_w[t * k + j] * y[h];
      if (y_all) memcpy(y_all + (n * k + j) * H, y, sizeof(double) * (size_t)H);
    }
    free(g);
  }
  return bad ? -1 : 0;
}

/* Expert intermediates of listed (token, expert) pairs, for localising a
 * mismatch: g, u, a [n, I] and y [n, H] of expert e on token t. */
EXPORT int oracle_expert_rows(const oracle_shape *sh, const uint16_t *x, const uint16_t *Wg,
                              const uint16_t *Wu, const uint16_t *Wd, const float *fWg,
                              const float *fWu, const float *fWd, int64_t n,
                              const int64_t *tokens, const int32_t *experts, double *g, double *u,
                              double *a, double *y) {
  ctx_t c;
  ctx_init(&c, sh, x, Wg, Wu, Wd, NULL, NULL, NULL, NULL);
  if (ctx_forward_quant(&c, fWg, fWu, fWd)) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t q = 0; q < n; ++q) {
    if (tokens[q] < 0 || tokens[q] >= sh->T || experts[q] < 0 || experts[q] >= sh->E) {
      bad = 1;
      continue;
    }
    expert_fwd(&c, tokens[q], experts[q], g + q * sh->I, u + q * sh->I, a + q * sh->I,
               y + q * sh->H);
  }
  return bad ? -1 : 0;
}

/* Backward for a list of tokens.
 *   gdot_j   = <dy_t, y(t, S_j)>                       (gradient wrt w_j)
 *   da       = w_j * dy_t . W_down[e]^T
 *   dg       = da * u * sigma(g) * (1 + g (1 - sigma(g)))   (d silu(g) u / dg)
 *   du       = da * silu(g)
 *   dx_t    += dg . W_gate[e]^T + du . W_up[e]^T
 * Router: w_j = p_{S_j} / P with P = sum_{S} p and p = softmax(l).  By the
 * chain rule through the renormalisation, dL/dp_e = (gdot_e - sum_i w_i gdot_i)/P
 * for kept e and 0 otherwise; then through the softmax (see below),
 * dL/dl_m = p_m dL/dp_m.
 * quant != 0: the backward GEMM operands dyw (=w dy) and W_down are quantised
 * along H, dg/du and W_gate/W_up along I, as MXFP8 (see the file header). */
EXPORT int oracle_backward_tokens(const oracle_shape *sh, const uint16_t *x, const float *logits,
                                  const int32_t *topk_idx, const double *topk_w, const uint16_t *Wg,
                                  const uint16_t *Wu, const uint16_t *Wd, const uint16_t *dy,
                                  int32_t quant, const float *qWg, const float *qWu,
                                  const float *qWd, const float *fWg, const float *fWu,
                                  const float *fWd, int64_t ntok, const int64_t *tokens, double *dx,
                                  double *d_logits, double *gdot_out) {
  const int H = sh->H, I = sh->I, E = sh->E, k = sh->k;
  if (quant && (!qWg || !qWu || !qWd || H % 32 || I % 32)) return -1;
  ctx_t c;
  ctx_init(&c, sh, x, Wg, Wu, Wd, dy, qWg, qWu, qWd);
  if (ctx_forward_quant(&c, fWg, fWu, fWd)) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t n = 0; n < ntok; ++n) {
    int64_t t = tokens[n];
    if (t < 0 || t >= sh->T) {
      bad = 1;
      continue;
    }
    double *buf = malloc(sizeof(double) * (size_t)(6 * I + 2 * H + 3 * E + 2 * k));
    double *g = buf, *u = g + I, *a = u + I, *da = a + I, *dg = da + I, *du = dg + I;
    double *y = du + I, *dyw = y + H, *p = dyw + H, *dp = p + E, *dl = dp + E;
    double *gd = dl + E, *wv = gd + k;
    int32_t sel[4096];
    const uint16_t *dyt = dy + t * H;
    for (int h = 0; h < H; ++h) dx[n * H + h] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[t * k + j];
      double w = topk_w[t * k + j];
      expert_fwd(&c, t, e, g, u, a, y);
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += bf(dyt[h]) * y[h];
      gd[j] = s;
      if (quant) { /* dA = w * (Q(dy) . Q(W_down)^T) */
        for (int h = 0; h < H; ++h) dyw[h] = bf(dyt[h]);
        mx_vec(dyw, H, 1);
      } else {
        for (int h = 0; h < H; ++h) dyw[h] = w * bf(dyt[h]);
      }
      for (int i = 0; i < I; ++i) {
        double acc = 0.0;
        if (quant) {
          const float *wd = qWd + ((int64_t)e * I + i) * H;
          for (int h = 0; h < H; ++h) acc += dyw[h] * (double)wd[h];
          acc *= w;
        } else {
          const uint16_t *wd = Wd + ((int64_t)e * I + i) * H;
          for (int h = 0; h < H; ++h) acc += dyw[h] * bf(wd[h]);
        }
        da[i] = acc;
      }
      for (int i = 0; i < I; ++i) {
        /* fp8_bwd: dSwiGLU reads the saved bf16 activations */
        const double gi = quant ? oracle_round_bf16(g[i]) : g[i];
        const double ui = quant ? oracle_round_bf16(u[i]) : u[i];
        double sg = sigmoid(gi);
        dg[i] = da[i] * ui * sg * (1.0 + gi * (1.0 - sg));
        du[i] = da[i] * silu(gi);
      }
      if (quant) {
        for (int i = 0; i < I; ++i) {
          dg[i] = oracle_round_bf16(dg[i]);
          du[i] = oracle_round_bf16(du[i]);
        }
        mx_vec(dg, I, 1);
        mx_vec(du, I, 1);
      }
      for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        if (quant) {
          const float *wg = qWg + ((int64_t)e * H + h) * I, *wu = qWu + ((int64_t)e * H + h) * I;
          for (int i = 0; i < I; ++i) acc += dg[i] * (double)wg[i] + du[i] * (double)wu[i];
        } else {
          const uint16_t *wg = Wg + ((int64_t)e * H + h) * I, *wu = Wu + ((int64_t)e * H + h) * I;
          for (int i = 0; i < I; ++i) acc += dg[i] * bf(wg[i]) + du[i] * bf(wu[i]);
        }
        dx[n * H + h] += acc;
      }
    }
    /* router */
    route_token(E, k, logits + t * E, sel, wv, p);
    double P = 0.0, gbar = 0.0;
    for (int j = 0; j < k; ++j) {
      P += p[sel[j]];
      gbar += wv[j] * gd[j];
    }
    for (int e = 0; e < E; ++e) dp[e] = 0.0;
    for (int j = 0; j < k; ++j) dp[sel[j]] = (gd[j] - gbar) / P;
    /* softmax backward: dL/dl_m = p_m (dL/dp_m - sum_e p_e dL/dp_e).  The sum is
     * sum_j (p_{S_j}/P)(gdot_j - gbar) = sum_j w_j gdot_j - gbar = 0 identically
     * (the kept weights sum to one), so it is left out rather than evaluated as
     * rounding noise; experts outside the kept set get an exact zero. */
    for (int e = 0; e < E; ++e) dl[e] = p[e] * dp[e];
    if (d_logits)
      for (int e = 0; e < E; ++e) d_logits[n * E + e] = dl[e];
    if (gdot_out)
      for (int j = 0; j < k; ++j) gdot_out[n * k + j] = gd[j];
    free(buf);
  }
  return bad ? -1 : 0;
}

/* Rows of expert e in token order (from the oracle's own dispatch). */
static int64_t expert_rows(const oracle_shape *sh, const int32_t *topk_idx, int e, int64_t *tok,
                           int32_t *choice) {
  int64_t n = 0;
  for (int64_t t = 0; t < sh->T; ++t)
    for (int j = 0; j < sh->k; ++j)
      if (topk_idx[t * sh->k + j] == e) {
        tok[n] = t;
        choice[n] = j;
        ++n;
      }
  return n;
}

/* Per-row backward intermediates of expert e over its rows: the two dW_down
 * operands (exact: a [n,I] and w dy [n,H]; quant: w a and dy), dg [n,I], du [n,I].
 * In quant mode dA's operands are quantised along H (matching
 * oracle_backward_tokens); the dW operands are quantised afterwards along tokens
 * by the caller. */
static void expert_rows_bwd(const ctx_t *c, int e, int64_t n, const int64_t *tok,
                            const int32_t *choice, const double *topk_w, int quant, double *A,
                            double *DYW, double *DG, double *DU) {
  const int H = c->sh->H, I = c->sh->I, k = c->sh->k;
  double *g = malloc(sizeof(double) * (size_t)(4 * I + H));
  double *u = g + I, *a = u + I, *da = a + I, *q = da + I;
  for (int64_t r = 0; r < n; ++r) {
    int64_t t = tok[r];
    double w = topk_w[t * k + choice[r]];
    expert_fwd(c, t, e, g, u, a, NULL);
    /* exact: dW_down operands a and w dy.  quant: w a and dy, and dA = w (Q(dy) . Q(W_down)^T) */
    const double ws = quant ? 1.0 : w;
    for (int h = 0; h < H; ++h) q[h] = ws * bf(c->dy[t * H + h]);
    for (int h = 0; h < H; ++h) DYW[r * H + h] = q[h];
    if (quant) mx_vec(q, H, 1);
    for (int i = 0; i < I; ++i) {
      double acc = 0.0;
      if (quant) {
        const float *wd = c->qWd + ((int64_t)e * I + i) * H;
        for (int h = 0; h < H; ++h) acc += q[h] * (double)wd[h];
        acc *= w;
      } else {
        const uint16_t *wd = c->Wd + ((int64_t)e * I + i) * H;
        for (int h = 0; h < H; ++h) acc += q[h] * bf(wd[h]);
      }
      da[i] = acc;
    }
    for (int i = 0; i < I; ++i) {
      if (quant) { /* bf16 tensors: saved g, u in; w*a, dg, du out */
        const double gi = oracle_round_bf16(g[i]), ui = oracle_round_bf16(u[i]);
        const double sg = sigmoid(gi);
        A[r * I + i] = oracle_round_bf16(w * a[i]);
        DG[r * I + i] = oracle_round_bf16(da[i] * ui * sg * (1.0 + gi * (1.0 - sg)));
        DU[r * I + i] = oracle_round_bf16(da[i] * silu(gi));
      } else {
        const double sg = sigmoid(g[i]);
        A[r * I + i] = a[i];
        DG[r * I + i] = da[i] * u[i] * sg * (1.0 + g[i] * (1.0 - sg));
        DU[r * I + i] = da[i] * silu(g[i]);
      }
    }
  }
  free(g);
}

/* Full weight gradients, one expert at a time over its rows in token order:
 *   dW_down[e] = sum_r a_r^T (w dy)_r,   dW_gate[e] = sum_r x_r^T dg_r,
 *   dW_up[e]   = sum_r x_r^T du_r.
 * Experts that received no token get exactly zero.  quant != 0: every operand
 * of these three GEMMs is quantised along tokens, blocks of 32 rows from the
 * expert's first row, zero-padded.  Outputs: dWg, dWu [E,H,I], dWd [E,I,H]. */
EXPORT int oracle_dw_full(const oracle_shape *sh, const uint16_t *x, const int32_t *topk_idx,
                          const double *topk_w, const uint16_t *Wg, const uint16_t *Wu,
                          const uint16_t *Wd, const uint16_t *dy, int32_t quant, const float *qWg,
                          const float *qWu, const float *qWd, const float *fWg, const float *fWu,
                          const float *fWd, double *dWg, double *dWu, double *dWd) {
  const int H = sh->H, I = sh->I, E = sh->E;
  ctx_t c;
  ctx_init(&c, sh, x, Wg, Wu, Wd, dy, qWg, qWu, qWd);
  if (ctx_forward_quant(&c, fWg, fWu, fWd)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int e = 0; e < E; ++e) {
    int64_t *tok = malloc(sizeof(int64_t) * (size_t)sh->T);
    int32_t *ch = malloc(sizeof(int32_t) * (size_t)sh->T);
    int64_t n = expert_rows(sh, topk_idx, e, tok, ch);
    double *A = malloc(sizeof(double) * (size_t)(n * I + 1));
    double *DYW = malloc(sizeof(double) * (size_t)(n * H + 1));
    double *DG = malloc(sizeof(double) * (size_t)(n * I + 1));
    double *DU = malloc(sizeof(double) * (size_t)(n * I + 1));
    double *X = malloc(sizeof(double) * (size_t)(n * H + 1));
    expert_rows_bwd(&c, e, n, tok, ch, topk_w, quant, A, DYW, DG, DU);
    for (int64_t r = 0; r < n; ++r)
      for (int h = 0; h < H; ++h) X[r * H + h] = bf(x[tok[r] * H + h]);
    if (quant) {
      for (int i = 0; i < I; ++i) {
        mx_vec(A + i, n, I);
        mx_vec(DG + i, n, I);
        mx_vec(DU + i, n, I);
      }
      for (int h = 0; h < H; ++h) {
        mx_vec(DYW + h, n, H);
        mx_vec(X + h, n, H);
      }
    }
    double *wd = dWd + (int64_t)e * I * H, *wg = dWg + (int64_t)e * H * I,
           *wu = dWu + (int64_t)e * H * I;
    memset(wd, 0, sizeof(double) * (size_t)I * H);
    memset(wg, 0, sizeof(double) * (size_t)H * I);
    memset(wu, 0, sizeof(double) * (size_t)H * I);
    for (int64_t r = 0; r < n; ++r) {
      for (int i = 0; i < I; ++i)
        for (int h = 0; h < H; ++h) wd[(int64_t)i * H + h] += A[r * I + i] * DYW[r * H + h];
      for (int h = 0; h < H; ++h)
        for (int i = 0; i < I; ++i) {
          wg[(int64_t)h * I + i] += X[r * H + h] * DG[r * I + i];
          wu[(int64_t)h * I + i] += X[r * H + h] * DU[r * I + i];
        }
    }
    free(tok);
    free(ch);
    free(A);
    free(DYW);
    free(DG);
    free(DU);
    free(X);
  }
  return 0;
}

/* Selected weight-gradient elements.  which: 0 = dW_gate[e,h,i] (r=h, c=i),
 * 1 = dW_up[e,h,i], 2 = dW_down[e,i,h] (r=i, c=h).  Each element is the sum
 * over expert e's rows in token order, as in oracle_dw_full; in quant mode the
 * two operand columns are quantised along tokens as there. */
EXPORT int oracle_dw_elements(const oracle_shape *sh, const uint16_t *x, const int32_t *topk_idx,
                              const double *topk_w, const uint16_t *Wg, const uint16_t *Wu,
                              const uint16_t *Wd, const uint16_t *dy, int32_t quant,
                              const float *qWg, const float *qWu, const float *qWd,
                              const float *fWg, const float *fWu, const float *fWd, int64_t nel,
                              const int32_t *which, const int32_t *ee, const int32_t *rr,
                              const int32_t *cc, double *val) {
  const int H = sh->H, I = sh->I, k = sh->k;
  ctx_t c;
  ctx_init(&c, sh, x, Wg, Wu, Wd, dy, qWg, qWu, qWd);
  if (ctx_forward_quant(&c, fWg, fWu, fWd)) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t q = 0; q < nel; ++q) {
    int e = ee[q], wh = which[q], r0 = rr[q], c0 = cc[q];
    if (e < 0 || e >= sh->E || wh < 0 || wh > 2) {
      bad = 1;
      continue;
    }
    int64_t *tok = malloc(sizeof(int64_t) * (size_t)sh->T);
    int32_t *ch = malloc(sizeof(int32_t) * (size_t)sh->T);
    int64_t n = expert_rows(sh, topk_idx, e, tok, ch);
    double *L = malloc(sizeof(double) * (size_t)(n + 1));
    double *R = malloc(sizeof(double) * (size_t)(n + 1));
    double *dyw = malloc(sizeof(double) * (size_t)(2 * H));
    double *xq = dyw + H;
    /* only column ci of g and u is needed: the same sums over h, in the same
     * order, as expert_fwd (or expert_fwd_mx) computes for every column */
    const int ci = (wh == 2) ? r0 : c0;
    const uint16_t *wg = Wg + (int64_t)e * H * I, *wu = Wu + (int64_t)e * H * I;
    for (int64_t r = 0; r < n; ++r) {
      int64_t t = tok[r];
      double w = topk_w[t * k + ch[r]];
      double gi = 0.0, ui = 0.0;
      if (c.fWg) {
        const float *fg = c.fWg + (int64_t)e * H * I, *fu = c.fWu + (int64_t)e * H * I;
        for (int h = 0; h < H; ++h) xq[h] = bf(x[t * H + h]);
        mx_vec(xq, H, 1);
        for (int h = 0; h < H; ++h) {
          gi += xq[h] * (double)fg[(int64_t)h * I + ci];
          ui += xq[h] * (double)fu[(int64_t)h * I + ci];
        }
      } else {
        for (int h = 0; h < H; ++h) {
          double xv = bf(x[t * H + h]);
          gi += xv * bf(wg[(int64_t)h * I + ci]);
          ui += xv * bf(wu[(int64_t)h * I + ci]);
        }
      }
      if (wh == 2) { /* dW_down[e, i=r0, h=c0] = sum a_i * (w dy)_h */
        if (quant) { /* operands w*a (a bf16 tensor) and dy */
          L[r] = oracle_round_bf16(w * silu(gi) * ui);
          R[r] = bf(dy[t * H + c0]);
        } else {
          L[r] = silu(gi) * ui;
          R[r] = w * bf(dy[t * H + c0]);
        }
      } else { /* dW_gate/up[e, h=r0, i=c0] = sum x_h * dg_i (du_i) */
        double da = 0.0;
        if (quant) {
          for (int h = 0; h < H; ++h) dyw[h] = bf(dy[t * H + h]);
          mx_vec(dyw, H, 1);
          const float *wd = qWd + ((int64_t)e * I + c0) * H;
          for (int h = 0; h < H; ++h) da += dyw[h] * (double)wd[h];
          da *= w;
        } else {
          for (int h = 0; h < H; ++h) dyw[h] = w * bf(dy[t * H + h]);
          const uint16_t *wd = Wd + ((int64_t)e * I + c0) * H;
          for (int h = 0; h < H; ++h) da += dyw[h] * bf(wd[h]);
        }
        if (quant) { /* saved bf16 activations in, a bf16 gradient out */
          gi = oracle_round_bf16(gi);
          ui = oracle_round_bf16(ui);
        }
        double sg = sigmoid(gi);
        L[r] = bf(x[t * H + r0]);
        R[r] = (wh == 0) ? da * ui * sg * (1.0 + gi * (1.0 - sg)) : da * silu(gi);
        if (quant) R[r] = oracle_round_bf16(R[r]);
      }
    }
    if (quant) {
      mx_vec(L, n, 1);
      mx_vec(R, n, 1);
    }
    double s = 0.0;
    for (int64_t r = 0; r < n; ++r) s += L[r] * R[r];
    val[q] = s;
    free(tok);
    free(ch);
    free(L);
    free(R);
    free(dyw);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Router projection: the learned router's linear layer, logits = x . W_r.    */
/* ------------------------------------------------------------------------- */

/* logits[t, e] = sum_h x[t, h] W_r[h, e]; x [T,H] and W_r [H,E] bf16; fp64 out. */
EXPORT int oracle_router_forward(int64_t T, int32_t H, int32_t E, const uint16_t *x,
                                 const uint16_t *Wr, double *logits) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    double *lt = logits + t * E;
    for (int e = 0; e < E; ++e) lt[e] = 0.0;
    for (int h = 0; h < H; ++h) {
      const double xv = bf(x[t * H + h]);
      const uint16_t *w = Wr + (int64_t)h * E;
      for (int e = 0; e < E; ++e) lt[e] += xv * bf(w[e]);
    }
  }
  return 0;
}

/* Backward of the router projection for an upstream gradient d_logits [T,E]:
 *   dW_r[h, e] = sum_t x[t, h] d_logits[t, e]     (fp64, [H,E])
 *   dx[t, h]   = sum_e d_logits[t, e] W_r[h, e]   (fp64, [T,H]; the router's
 *                contribution to the layer input's gradient). */
EXPORT int oracle_router_backward(int64_t T, int32_t H, int32_t E, const uint16_t *x,
                                  const uint16_t *Wr, const double *d_logits, double *dWr,
                                  double *dx) {
#pragma omp parallel for schedule(static)
  for (int h = 0; h < H; ++h) {
    double *dw = dWr + (int64_t)h * E;
    for (int e = 0; e < E; ++e) dw[e] = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const double xv = bf(x[t * H + h]);
      const double *g = d_logits + t * E;
      for (int e = 0; e < E; ++e) dw[e] += xv * g[e];
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double *g = d_logits + t * E;
    for (int h = 0; h < H; ++h) {
      const uint16_t *w = Wr + (int64_t)h * E;
      double acc = 0.0;
      for (int e = 0; e < E; ++e) acc += g[e] * bf(w[e]);
      dx[t * H + h] = acc;
    }
  }
  return 0;
}
