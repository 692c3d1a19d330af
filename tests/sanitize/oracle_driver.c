/*
 * oracle_driver.c -- runs every entry point of oracle/moe_oracle.c on small seeded problems in a
 * build with AddressSanitizer and UndefinedBehaviorSanitizer (tests/test_sanitizers.py compiles
 * it together with the oracle).  Any out-of-bounds access, use of freed memory, leak or undefined
 * operation aborts the run; the checks below only make sure every path really executes.
 * Test infrastructure: the oracle's prototypes are restated here (the oracle has no header).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const uint8_t *codes;
  const uint16_t *scales;
  const uint16_t *biases;
  int32_t rows, cols, bits;
} oracle_proj;

double oracle_f16(uint16_t h);
double oracle_bf16(uint16_t b);
uint32_t oracle_code(const uint8_t *row, int32_t bits, int64_t c);
double oracle_weight(const oracle_proj *p, int64_t r, int64_t c);
int oracle_moe_token(int32_t din, int32_t dff, int32_t top_k, const oracle_proj *gate,
                     const oracle_proj *up, const oracle_proj *down, const float *scores,
                     int32_t n_shared, int32_t dff_shared, const oracle_proj *sh_gate,
                     const oracle_proj *sh_up, const oracle_proj *sh_down,
                     const uint16_t *gate_vec, const uint16_t *x_bf16, const void *resid,
                     int32_t resid_kind, double *out, const int32_t *rows, int32_t n_rows);
int32_t oracle_route_invert(const int32_t *ids, int32_t m, int32_t k, int32_t n_experts,
                            int32_t *uniq, int32_t *offs, int32_t *pairs);
void oracle_router(const float *logits, int32_t n_experts, int32_t k, int32_t *ids,
                   float *scores);
uint16_t oracle_round_bf16(double y);
void oracle_rmsnorm_bf16(const float *v, int32_t n, const uint16_t *gamma, float eps,
                         uint16_t *x);
void oracle_gemv_bf16(const uint16_t *W, const uint16_t *x, int32_t m, int32_t n_out,
                      int32_t n_in, double *y);

static uint64_t state = 0x5EEDull;
static uint32_t next_u32(void) {  /* a plain 64-bit LCG, high half */
  state = state * 6364136223846793005ull + 1442695040888963407ull;
  return (uint32_t)(state >> 32);
}

#define CHECK(c)                                                        \
  do {                                                                  \
    if (!(c)) {                                                         \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c);   \
      return 1;                                                         \
    }                                                                   \
  } while (0)

/* One expert projection with exactly rows * cols * bits / 8 code bytes (no slack), codes drawn at
 * random and packed LSB first; scales about 0.01 (fp16 0x211F), biases about -0.08 (0xAD1F). */
typedef struct {
  oracle_proj p;
  uint8_t *codes;
  uint16_t *scales, *biases;
  uint8_t *plain;  /* the drawn codes, [rows][cols] */
} proj_buf;

static int make_proj(proj_buf *b, int32_t rows, int32_t cols, int32_t bits) {
  const int64_t rb = (int64_t)cols * bits / 8, g = cols / 64;
  b->codes = (uint8_t *)calloc((size_t)(rows * rb), 1);
  b->scales = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(rows * g));
  b->biases = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(rows * g));
  b->plain = (uint8_t *)malloc((size_t)rows * (size_t)cols);
  if (!b->codes || !b->scales || !b->biases || !b->plain) return 1;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < cols; ++c) {
      const uint32_t q = next_u32() & ((1u << bits) - 1u);
      b->plain[r * cols + c] = (uint8_t)q;
      for (int32_t t = 0; t < bits; ++t) {
        const int64_t bit = c * bits + t;
        if ((q >> t) & 1u) b->codes[r * rb + bit / 8] |= (uint8_t)(1u << (bit % 8));
      }
    }
    for (int64_t j = 0; j < g; ++j) {
      b->scales[r * g + j] = (uint16_t)(0x211F + (next_u32() & 0xff));
      b->biases[r * g + j] = (uint16_t)(0xAD1F + (next_u32() & 0xff));
    }
  }
  b->p.codes = b->codes;
  b->p.scales = b->scales;
  b->p.biases = b->biases;
  b->p.rows = rows;
  b->p.cols = cols;
  b->p.bits = bits;
  return 0;
}

static void free_proj(proj_buf *b) {
  free(b->codes);
  free(b->scales);
  free(b->biases);
  free(b->plain);
}

static uint16_t bf16_of(double v) { return oracle_round_bf16(v); }

int main(void) {
  /* codes read back at every width, every column of the last row (the end of the buffer) */
  const int32_t widths[3] = {4, 6, 8};
  for (int w = 0; w < 3; ++w) {
    proj_buf b;
    CHECK(make_proj(&b, 3, 192, widths[w]) == 0);
    for (int64_t r = 0; r < 3; ++r)
      for (int64_t c = 0; c < 192; ++c)
        CHECK(oracle_code(b.codes + r * 192 * widths[w] / 8, widths[w], c) == b.plain[r * 192 + c]);
    CHECK(isfinite(oracle_weight(&b.p, 2, 191)));
    free_proj(&b);
  }

  /* one token: 2 routed slots (6-bit gate/up, 4-bit down), 1 gated 8-bit shared expert, every
   * row and then a list of rows, bf16 and fp32 residuals */
  enum { DIN = 128, DFF = 64, K = 2, DSH = 128 };
  proj_buf g[K], u[K], d[K], sg, su, sd;
  oracle_proj pg[K], pu[K], pd[K];
  for (int k = 0; k < K; ++k) {
    CHECK(make_proj(&g[k], DFF, DIN, 6) == 0 && make_proj(&u[k], DFF, DIN, 6) == 0 &&
          make_proj(&d[k], DIN, DFF, 4) == 0);
    pg[k] = g[k].p;
    pu[k] = u[k].p;
    pd[k] = d[k].p;
  }
  CHECK(make_proj(&sg, DSH, DIN, 8) == 0 && make_proj(&su, DSH, DIN, 8) == 0 &&
        make_proj(&sd, DIN, DSH, 8) == 0);
  uint16_t x[DIN], gv[DIN], r16[DIN];
  float r32[DIN];
  for (int c = 0; c < DIN; ++c) {
    x[c] = bf16_of(((int)(next_u32() % 2001) - 1000) / 500.0);
    gv[c] = bf16_of(((int)(next_u32() % 2001) - 1000) / 50000.0);
    r32[c] = (float)(((int)(next_u32() % 2001) - 1000) / 250.0);
    r16[c] = bf16_of(r32[c]);
  }
  const float scores[K] = {0.75f, 0.25f};
  double out[DIN], out_rows[3];
  const int32_t rows[3] = {0, 77, DIN - 1};
  CHECK(oracle_moe_token(DIN, DFF, K, pg, pu, pd, scores, 1, DSH, &sg.p, &su.p, &sd.p, gv, x, r16,
                         0, out, NULL, 0) == 0);
  CHECK(oracle_moe_token(DIN, DFF, K, pg, pu, pd, scores, 1, DSH, &sg.p, &su.p, &sd.p, gv, x, r32,
                         1, out_rows, rows, 3) == 0);
  for (int c = 0; c < DIN; ++c) CHECK(isfinite(out[c]));
  for (int t = 0; t < 3; ++t) CHECK(isfinite(out_rows[t]));
  /* a shape mismatch is refused */
  CHECK(oracle_moe_token(DIN, DFF + 64, K, pg, pu, pd, scores, 0, 0, NULL, NULL, NULL, NULL, x,
                         r16, 0, out, NULL, 0) == -1);
  for (int k = 0; k < K; ++k) {
    free_proj(&g[k]);
    free_proj(&u[k]);
    free_proj(&d[k]);
  }
  free_proj(&sg);
  free_proj(&su);
  free_proj(&sd);

  /* route inversion with out-of-range ids; router; RMSNorm; GEMV */
  enum { M = 5, KR = 3, E = 7 };
  int32_t ids[M * KR], uniq[M * KR], offs[M * KR + 1], pairs[M * KR];
  int valid = 0;
  for (int p = 0; p < M * KR; ++p) {
    ids[p] = (int32_t)(next_u32() % (E + 2)) - 1;  /* -1 .. E */
    valid += ids[p] >= 0 && ids[p] < E;
  }
  const int32_t U = oracle_route_invert(ids, M, KR, E, uniq, offs, pairs);
  CHECK(U >= 0 && U <= E && offs[U] == valid);
  float logits[E], sc[E];
  int32_t top[E];
  for (int e = 0; e < E; ++e) logits[e] = (float)(next_u32() % 5);  /* ties on purpose */
  oracle_router(logits, E, E, top, sc);
  for (int a = 0; a < E; ++a)
    for (int b2 = a + 1; b2 < E; ++b2) CHECK(top[a] != top[b2]);
  float v[DIN];
  uint16_t gamma[DIN], xn[DIN];
  for (int c = 0; c < DIN; ++c) {
    v[c] = r32[c];
    gamma[c] = bf16_of(1.0 + ((int)(next_u32() % 201) - 100) / 500.0);
  }
  oracle_rmsnorm_bf16(v, DIN, gamma, 1e-6f, xn);
  enum { GM = 3, GO = 5, GI = 64 };
  uint16_t W[GO * GI], xg[GM * GI];
  double y[GM * GO];
  for (int i = 0; i < GO * GI; ++i) W[i] = bf16_of(((int)(next_u32() % 201) - 100) / 1000.0);
  for (int i = 0; i < GM * GI; ++i) xg[i] = bf16_of(((int)(next_u32() % 201) - 100) / 100.0);
  oracle_gemv_bf16(W, xg, GM, GO, GI, y);
  for (int i = 0; i < GM * GO; ++i) CHECK(isfinite(y[i]));
  CHECK(oracle_f16(0x3C00) == 1.0 && oracle_bf16(0x3F80) == 1.0);
  printf("oracle sanitizer run ok\n");
  return 0;
}
