/*
 * moe_oracle.c -- fp64 CPU oracle of the single-token decode MoE expert block.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  It shares no code, header,
 * table or helper with the CUDA path and includes nothing from it.
 *
 * What it computes (one token, every step written out in its plainest form, in fp64):
 *
 *   unpack   q[r][c]  = bits [c*b, c*b+b) of packed row r, read LSB first
 *            (canonical layout: row-major codes, little-endian bit stream per row)
 *   dequant  w[r][c]  = scale[r][c/64] * q[r][c] + bias[r][c/64]        (affine, group 64)
 *   kernel A g_j = sum_c w_gate[j][c] x_c ;  u_j = sum_c w_up[j][c] x_c
 *            act_j = silu(g_j) * u_j ,  silu(z) = z / (1 + exp(-z))
 *            -- "two-kernel decode-MoE that beats gather_qmm", What changed, step 2
 *               (A: gate/up + swiglu into act_g[K, Dff])
 *   kernel B y_k[i] = sum_j w_down,k[i][j] act_k[j]
 *            routed[i] = sum_k score_k * y_k[i], k in the order the ids are given
 *            -- same page, step 2 (B: down * score, summed over K)
 *   tail     out[i] = resid[i] + (routed[i] + shared_scalar * shared[i])
 *            shared[i] = sum over shared experts of their down outputs
 *            shared_scalar = sigmoid(x . g) when a gate vector is given, else 1
 *            -- "Red Lite dev39 -- fused expert tail", Change (routed = sum_e
 *               weights[e] tmp[e][i] in the pool's order, then x = resid +
 *               (routed + shared * scalar))
 *
 *   norm     (a stack with the next layer's RMSNorm folded in) the next layer's input
 *            x_c = gamma_c * v_c / sqrt((1/n) sum_j v_j^2 + eps), rounded to bf16
 *            -- "Red Lite dev39 -- fused expert tail", Measurements (the tail variant that
 *               also folded in the next layer's RMSNorm); see oracle_rmsnorm_bf16
 *
 * No intermediate value of the block is rounded: codes are exact integers, fp16 and bf16 inputs
 * convert to double exactly, and every sum runs left to right in double.  The norm's output is a
 * bf16 code: computed in double and rounded once (oracle_rmsnorm_bf16).
 * Pins: tests/test_oracle_pins.py.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const uint8_t *codes;    /* [rows][cols*bits/8]: packed codes of one expert's projection */
  const uint16_t *scales;  /* [rows][cols/64]: fp16 bit patterns */
  const uint16_t *biases;  /* [rows][cols/64]: fp16 bit patterns */
  int32_t rows, cols, bits;
} oracle_proj;

/* IEEE binary16 bit pattern -> double (exact). */
double oracle_f16(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16 bit pattern -> double (exact): bf16 is the upper half of an IEEE binary32. */
double oracle_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Code c of a packed row: bits [c*bits, c*bits + bits) of the row's bit stream, where bit t of
 * the stream is bit (t mod 8) of byte (t / 8) -- a little-endian, LSB-first stream. */
uint32_t oracle_code(const uint8_t *row, int32_t bits, int64_t c) {
  uint32_t q = 0;
  for (int32_t t = 0; t < bits; ++t) {
    int64_t bit = c * bits + t;
    q |= (uint32_t)((row[bit >> 3] >> (bit & 7)) & 1u) << t;
  }
  return q;
}

/* Dequantized weight w[r][c] = scale * q + bias of its group of 64 columns. */
double oracle_weight(const oracle_proj *p, int64_t r, int64_t c) {
  const int64_t groups = p->cols / 64;
  const int64_t rowbytes = (int64_t)p->cols * p->bits / 8;
  const double scale = oracle_f16(p->scales[r * groups + c / 64]);
  const double bias = oracle_f16(p->biases[r * groups + c / 64]);
  const double q = (double)oracle_code(p->codes + r * rowbytes, p->bits, c);
  return scale * q + bias;
}

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

double oracle_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* y[r] = sum_c w[r][c] * v[c] for the listed rows (all rows when rows == NULL). */
void oracle_matvec(const oracle_proj *p, const double *v, double *y, const int32_t *rows,
                   int32_t n_rows) {
  const int32_t n = rows ? n_rows : p->rows;
  for (int32_t t = 0; t < n; ++t) {
    const int64_t r = rows ? rows[t] : t;
    double acc = 0.0;
    for (int64_t c = 0; c < p->cols; ++c) acc += oracle_weight(p, r, c) * v[c];
    y[rows ? t : r] = acc;
  }
}

/* act_j = silu(gate_j . x) * (up_j . x) for every row j of one expert (kernel A). */
void oracle_expert_act(const oracle_proj *gate, const oracle_proj *up, const double *x,
                       double *act) {
  const int32_t dff = gate->rows;
  double *g = (double *)malloc(sizeof(double) * dff);
  double *u = (double *)malloc(sizeof(double) * dff);
  oracle_matvec(gate, x, g, NULL, 0);
  oracle_matvec(up, x, u, NULL, 0);
  for (int32_t j = 0; j < dff; ++j) act[j] = oracle_silu(g[j]) * u[j];
  free(g);
  free(u);
}

/* sigmoid(x . g) over din elements; g is bf16. */
double oracle_shared_scalar(const double *x, const uint16_t *gate_vec, int32_t din) {
  double dot = 0.0;
  for (int32_t c = 0; c < din; ++c) dot += x[c] * oracle_bf16(gate_vec[c]);
  return oracle_sigmoid(dot);
}

/* Whole block for one token.  x is bf16 [din]; resid is bf16 (resid_kind 0) or fp32 (1) [din];
 * out is double [n_rows] (rows listed) or [din] (rows == NULL).  The k-th routed slot uses
 * gate[k], up[k], down[k] (the expert that ids[k] names, gathered by the caller) and scores[k].
 * Returns 0, or -1 on a shape mismatch or allocation failure. */
int oracle_moe_token(int32_t din, int32_t dff, int32_t top_k, const oracle_proj *gate,
                     const oracle_proj *up, const oracle_proj *down, const float *scores,
                     int32_t n_shared, int32_t dff_shared, const oracle_proj *sh_gate,
                     const oracle_proj *sh_up, const oracle_proj *sh_down,
                     const uint16_t *gate_vec, const uint16_t *x_bf16, const void *resid,
                     int32_t resid_kind, double *out, const int32_t *rows, int32_t n_rows) {
  for (int32_t k = 0; k < top_k; ++k)
    if (gate[k].rows != dff || gate[k].cols != din || up[k].rows != dff || up[k].cols != din ||
        down[k].rows != din || down[k].cols != dff)
      return -1;
  for (int32_t s = 0; s < n_shared; ++s)
    if (sh_gate[s].rows != dff_shared || sh_gate[s].cols != din || sh_up[s].rows != dff_shared ||
        sh_up[s].cols != din || sh_down[s].rows != din || sh_down[s].cols != dff_shared)
      return -1;
  const int32_t n_out = rows ? n_rows : din;
  double *x = (double *)malloc(sizeof(double) * din);
  double *routed = (double *)calloc(n_out, sizeof(double));
  double *shared = (double *)calloc(n_out, sizeof(double));
  double *y = (double *)malloc(sizeof(double) * n_out);
  const int32_t dff_max = dff > dff_shared ? dff : dff_shared;
  double *act = (double *)malloc(sizeof(double) * (dff_max > 0 ? dff_max : 1));
  if (!x || !routed || !shared || !y || !act) {
    free(x); free(routed); free(shared); free(y); free(act);
    return -1;
  }
  for (int32_t c = 0; c < din; ++c) x[c] = oracle_bf16(x_bf16[c]);

  for (int32_t k = 0; k < top_k; ++k) {          /* routed experts, in the given slot order */
    oracle_expert_act(&gate[k], &up[k], x, act);
    oracle_matvec(&down[k], act, y, rows, n_rows);
    for (int32_t t = 0; t < n_out; ++t) routed[t] += (double)scores[k] * y[t];
  }
  for (int32_t s = 0; s < n_shared; ++s) {       /* shared experts, summed */
    oracle_expert_act(&sh_gate[s], &sh_up[s], x, act);
    oracle_matvec(&sh_down[s], act, y, rows, n_rows);
    for (int32_t t = 0; t < n_out; ++t) shared[t] += y[t];
  }
  const double scalar = gate_vec ? oracle_shared_scalar(x, gate_vec, din) : 1.0;
  for (int32_t t = 0; t < n_out; ++t) {
    const int32_t i = rows ? rows[t] : t;
    const double r = resid_kind == 0 ? oracle_bf16(((const uint16_t *)resid)[i])
                                     : (double)((const float *)resid)[i];
    out[t] = r + (routed[t] + scalar * shared[t]);
  }
  free(x); free(routed); free(shared); free(y); free(act);
  return 0;
}

/* Route inversion for m tokens of k routed slots each: the distinct valid expert ids in
 * ascending order, and for each of them the (token, slot) pairs whose id names it, written as
 * p = token * k + slot in ascending order.  Ids outside [0, n_experts) belong to no expert.
 * This is the grouping of the routers' top-k pools ("Red Lite dev39 -- fused expert tail",
 * Change) by expert, which lets a batch of tokens read each selected expert once.
 * Writes uniq[U], offs[U + 1] (the pairs of uniq[u] are pairs[offs[u]] .. pairs[offs[u + 1] - 1])
 * and pairs[offs[U]]; returns U.  Plain definition: one pass over the pairs per expert id. */
int32_t oracle_route_invert(const int32_t *ids, int32_t m, int32_t k, int32_t n_experts,
                            int32_t *uniq, int32_t *offs, int32_t *pairs) {
  int32_t u = 0, n = 0;
  offs[0] = 0;
  for (int32_t e = 0; e < n_experts; ++e) {
    int32_t found = 0;
    for (int32_t p = 0; p < m * k; ++p) {
      if (ids[p] == e) {
        pairs[n++] = p;
        found = 1;
      }
    }
    if (found) {
      uniq[u++] = e;
      offs[u] = n;
    }
  }
  return u;
}

/* Router of one token: the k largest of n_experts logits (fp32), larger first and, between equal
 * logits, the lower expert id first; scores are the softmax of the chosen logits over those k
 * ("Red Lite dev39 -- fused expert tail": the GPU-routed decode takes a top-k pool with weights
 * before the expert tail).  The ids are decided on the fp32 values as given (comparisons only);
 * the scores are computed in double and rounded to fp32.  Plain definition: k passes, each
 * taking the best remaining logit. */
void oracle_router(const float *logits, int32_t n_experts, int32_t k, int32_t *ids,
                   float *scores) {
  for (int32_t t = 0; t < k; ++t) {
    int32_t best = -1;
    for (int32_t e = 0; e < n_experts; ++e) {
      int32_t taken = 0;
      for (int32_t q = 0; q < t; ++q) taken |= ids[q] == e;
      if (taken) continue;
      if (best < 0 || logits[e] > logits[best]) best = e;  /* ties keep the lower id */
    }
    ids[t] = best;
  }
  double mx = -INFINITY, sum = 0.0;
  for (int32_t t = 0; t < k; ++t) mx = fmax(mx, (double)logits[ids[t]]);
  for (int32_t t = 0; t < k; ++t) sum += exp((double)logits[ids[t]] - mx);
  for (int32_t t = 0; t < k; ++t) scores[t] = (float)(exp((double)logits[ids[t]] - mx) / sum);
}


/* The bf16 nearest to y, ties to even (bit pattern).  bf16 keeps 8 significant bits, so y is
 * rounded at the spacing 2^(e-8) of its binade [2^(e-1), 2^e), never finer than the subnormal
 * spacing 2^-133; a value that rounds beyond the largest finite bf16 becomes an infinity. */
uint16_t oracle_round_bf16(double y) {
  if (isnan(y)) return 0x7fc0;
  const uint16_t sign = signbit(y) ? 0x8000 : 0;
  if (isinf(y)) return sign | 0x7f80;
  if (y == 0.0) return sign;
  int e;
  frexp(y, &e);
  int s = e - 8;
  if (s < -133) s = -133;
  const double q = ldexp(nearbyint(ldexp(y, -s)), s);  /* nearbyint: to nearest, ties to even */
  if (fabs(q) > FLT_MAX) return sign | 0x7f80;
  const float f = (float)q;                           /* exact: at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* The next layer's input from a layer's fp32 output v when the RMSNorm is folded into the tail
 * ("Red Lite dev39 -- fused expert tail", Measurements: the reverted tail that also folded in the
 * next layer's RMSNorm).  The page names the step without a formula; this is the usual RMSNorm,
 *   x_c = gamma_c * v_c * r,   r = 1 / sqrt((1/n) sum_j v_j^2 + eps),
 * computed in double and rounded once, at the end, to the nearest bf16 (ties to even).
 * v fp32 [n]; gamma bf16 [n]; x receives bf16 bit patterns [n]. */
void oracle_rmsnorm_bf16(const float *v, int32_t n, const uint16_t *gamma, float eps,
                         uint16_t *x) {
  double ss = 0.0;
  for (int32_t c = 0; c < n; ++c) ss += (double)v[c] * (double)v[c];
  const double r = 1.0 / sqrt(ss / n + (double)eps);
  for (int32_t c = 0; c < n; ++c) x[c] = oracle_round_bf16(oracle_bf16(gamma[c]) * ((double)v[c] * r));
}

/* Dense bf16 decode GEMV, the attention projections that "Measure attention projections instead
 * of serving them, and record the amortisation trap" measures at 1, 8 and 32 rows:
 *   y[t][o] = sum_i W[o][i] * x[t][i]
 * W bf16 [n_out][n_in] row-major, x bf16 [m][n_in], y double [m][n_out]; plain loops in double,
 * every sum left to right. */
void oracle_gemv_bf16(const uint16_t *W, const uint16_t *x, int32_t m, int32_t n_out,
                      int32_t n_in, double *y) {
  for (int32_t t = 0; t < m; ++t)
    for (int32_t o = 0; o < n_out; ++o) {
      double acc = 0.0;
      for (int32_t i = 0; i < n_in; ++i)
        acc += oracle_bf16(W[(int64_t)o * n_in + i]) * oracle_bf16(x[(int64_t)t * n_in + i]);
      y[(int64_t)t * n_out + o] = acc;
    }
}
