/*
 * Sanitizer driver for the oracle (test infrastructure): built together with
 * oracle/attn_oracle.c under AddressSanitizer and UndefinedBehaviorSanitizer,
 * it runs every exported oracle function on small problems whose buffers are
 * heap blocks of exactly the size the call may touch, including the edge
 * shapes (one key, one feature, causal and not, the last head and row), so an
 * access one element past a buffer or an undefined operation stops the run.
 * It also checks that the rows API returns the full evaluation's rows bit for
 * bit. Exit status: 0 when every check passed.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

int kb_oracle_attn(const double*, const double*, const double*, double*, int64_t, int64_t, int64_t, int64_t, int,
                   double);
int kb_oracle_lse(const double*, const double*, double*, int64_t, int64_t, int64_t, int, double);
int kb_oracle_attn_rows(const double*, const double*, const double*, double*, int64_t, int64_t, int64_t, int, double,
                        const int64_t*, const int64_t*, int64_t);
int kb_oracle_copy(float*, const float*, int64_t);
int kb_oracle_fill(float*, float, int64_t);
int kb_oracle_sum(const float*, int64_t, double*);
int kb_oracle_triad(float*, const float*, const float*, float, int64_t);
int kb_oracle_q15_exp_table(uint16_t*);
int kb_oracle_attn_q15(const int16_t*, const int16_t*, const int16_t*, int16_t*, int64_t, int64_t, int64_t, int,
                       double);

static int failures = 0;
#define CHECK(c)                                                      \
  do {                                                                \
    if (!(c)) {                                                       \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      ++failures;                                                     \
    }                                                                 \
  } while (0)

static uint64_t rng = 88172645463325252ull;
static double uniform(void) { /* xorshift64, U[-1, 1) */
  rng ^= rng << 13;
  rng ^= rng >> 7;
  rng ^= rng << 17;
  return (double)(rng >> 11) / 4503599627370496.0 - 1.0;
}

static double* drand_block(int64_t n) {
  double* p = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
  for (int64_t i = 0; i < n; ++i) p[i] = uniform();
  return p;
}

static void attention_shapes(void) {
  const int64_t shapes[][4] = {{1, 1, 1, 1}, {1, 1, 1, 7}, {1, 2, 5, 1}, {2, 3, 17, 4}, {1, 1, 64, 32}, {3, 1, 70, 3}};
  for (size_t t = 0; t < sizeof shapes / sizeof shapes[0]; ++t) {
    const int64_t B = shapes[t][0], H = shapes[t][1], S = shapes[t][2], d = shapes[t][3], N = B * H;
    double *q = drand_block(N * S * d), *k = drand_block(N * S * d), *v = drand_block(N * S * d);
    double* o = (double*)malloc((size_t)(N * S * d) * sizeof(double));
    double* lse = (double*)malloc((size_t)(N * S) * sizeof(double));
    for (int causal = 0; causal < 2; ++causal) {
      CHECK(kb_oracle_attn(q, k, v, o, B, H, S, d, causal, 0.7) == 0);
      for (int64_t i = 0; i < N * S * d; ++i) CHECK(isfinite(o[i]));
      CHECK(kb_oracle_lse(q, k, lse, N, S, d, causal, 0.7) == 0);
      for (int64_t i = 0; i < N * S; ++i) CHECK(isfinite(lse[i]));
      /* the first and last row of the first and last head, plus one in the middle */
      int64_t heads[5] = {0, 0, N - 1, N - 1, N / 2}, rows[5] = {0, S - 1, 0, S - 1, S / 2};
      double* r = (double*)malloc((size_t)(5 * d) * sizeof(double));
      CHECK(kb_oracle_attn_rows(q, k, v, r, N, S, d, causal, 0.7, heads, rows, 5) == 0);
      for (int e = 0; e < 5; ++e)
        CHECK(memcmp(r + e * d, o + (heads[e] * S + rows[e]) * d, (size_t)d * sizeof(double)) == 0);
      free(r);
    }
    /* rejected arguments touch nothing */
    CHECK(kb_oracle_attn(q, k, v, o, B, H, 0, d, 0, 0.7) != 0);
    CHECK(kb_oracle_attn(q, k, v, o, B, H, S, d, 0, NAN) != 0);
    int64_t bad_head = N, zero = 0;
    CHECK(kb_oracle_attn_rows(q, k, v, o, N, S, d, 0, 0.7, &bad_head, &zero, 1) != 0);
    free(q);
    free(k);
    free(v);
    free(o);
    free(lse);
  }
}

static void q15_shapes(void) {
  uint16_t* tab = (uint16_t*)malloc(64 * sizeof(uint16_t));
  CHECK(kb_oracle_q15_exp_table(tab) == 0 && tab[0] == 32768u);
  for (int f = 1; f < 64; ++f) CHECK(tab[f] < tab[f - 1] && tab[f] > 16384u);
  free(tab);
  const int64_t shapes[][3] = {{1, 1, 1}, {1, 33, 5}, {2, 70, 8}, {1, 64, 32}};
  for (size_t t = 0; t < sizeof shapes / sizeof shapes[0]; ++t) {
    const int64_t N = shapes[t][0], S = shapes[t][1], d = shapes[t][2], n = N * S * d;
    int16_t *q = (int16_t*)malloc((size_t)n * 2), *k = (int16_t*)malloc((size_t)n * 2),
            *v = (int16_t*)malloc((size_t)n * 2), *o = (int16_t*)malloc((size_t)n * 2);
    for (int64_t i = 0; i < n; ++i) {
      q[i] = (int16_t)(uniform() * 32767.0);
      k[i] = (int16_t)(uniform() * 32767.0);
      v[i] = (int16_t)(uniform() * 32767.0);
    }
    /* extremes of the format: full-scale inputs saturate nothing they should not */
    q[0] = -32768;
    k[n - 1] = 32767;
    v[n - 1] = -32768;
    for (int causal = 0; causal < 2; ++causal)
      CHECK(kb_oracle_attn_q15(q, k, v, o, N, S, d, causal, 1.0 / sqrt((double)d)) == 0);
    CHECK(kb_oracle_attn_q15(q, k, v, o, N, S, d, 0, 0.0) != 0);
    free(q);
    free(k);
    free(v);
    free(o);
  }
}

static void stream_kernels(void) {
  const int64_t lens[] = {0, 1, 3, 4, 1001};
  for (size_t t = 0; t < sizeof lens / sizeof lens[0]; ++t) {
    const int64_t n = lens[t];
    float *a = (float*)malloc((size_t)(n > 0 ? n : 1) * 4), *b = (float*)malloc((size_t)(n > 0 ? n : 1) * 4),
          *c = (float*)malloc((size_t)(n > 0 ? n : 1) * 4);
    for (int64_t i = 0; i < n; ++i) {
      b[i] = (float)uniform();
      c[i] = (float)uniform();
    }
    double sum = -1.0;
    CHECK(kb_oracle_triad(a, b, c, 3.0f, n) == 0);
    CHECK(kb_oracle_copy(a, b, n) == 0);
    CHECK(kb_oracle_fill(a, 2.5f, n) == 0);
    CHECK(kb_oracle_sum(a, n, &sum) == 0 && sum == 2.5 * (double)n);
    free(a);
    free(b);
    free(c);
  }
}

int main(void) {
  attention_shapes();
  q15_shapes();
  stream_kernels();
  if (failures) fprintf(stderr, "%d checks failed\n", failures);
  else printf("oracle sanitizer driver: all checks passed\n");
  return failures ? 1 : 0;
}
