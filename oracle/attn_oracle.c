/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY: the plain CPU oracle.
 *
 * This file is the slow, obviously-correct restatement of what the attention
 * library computes. It is used only by the tests, by the smoke check and by
 * the benchmark's CPU-baseline leg. No product code path links, loads or calls
 * it, and it shares no code, header or table with the CUDA library.
 *
 * Everything is single-threaded, in double precision, written as straight
 * loops that follow the mathematical definition with no blocking, fusion or
 * reordering. It is built with -ffp-contract=off so that x86_64 and aarch64
 * hosts produce the same bits.
 *
 * Sources (web pages):
 *  - "kbench -- Transformer Attention Micro-benchmark Harness",
 *    section "Implementation details / The three GPU kernels": every kernel
 *    computes O = softmax(Q K^T / sqrt(d)) V over a flattened (batch*heads)
 *    axis, laid out [head, seq, dim] row-major.
 *  - same page, section "CPU reference + cache profiling": a golden reference
 *    that every target is diffed against.
 *  - same page, sequence diagram "One MCU measurement": the request carries a
 *    causal flag next to seq and dim.
 *  - TileOPs "Hardware Microbenchmarks" README, section "HBM Bandwidth" and
 *    "Methodology": the STREAM Triad a[i] = b[i] + s*c[i], and the copy,
 *    read-only and write-only reference kernels beside it.
 *
 * Readings where the pages are silent:
 *  - causal: key j is visible to query i iff j <= i;
 *  - the scale is a parameter; it multiplies the raw dot product before the
 *    mask and before the row maximum (the pages fix it to 1/sqrt(d));
 *  - the row maximum is subtracted before exp; this leaves the mathematical
 *    result unchanged and keeps exp finite for large scores;
 *  - Triad rounds b + s*c once (a fused multiply-add), which is what a CUDA
 *    compiler emits for that expression by default.
 *
 * Parity status: pinned. The attention functions are pinned by a
 * high-precision brute-force evaluation on tiny inputs and by closed-form
 * invariants; the Triad is pinned by exact rational arithmetic and by the
 * STREAM constant check; copy, fill and sum by exact small-integer cases.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define KB_ORACLE_OK 0
#define KB_ORACLE_BAD_ARG 1
#define KB_ORACLE_NO_MEMORY 4

/*
 * Steps 1-3 for one query row of one head, as written on the kbench page
 * (one query row at a time):
 *   1. score s_j = scale * sum_c q[n,i,c] * k[n,j,c]   for every key j
 *   2. causal: keys j > i are left out (probability exactly 0)
 *   3. m = max_j s_j over the visible keys
 *   q, k : [N, S, d] row-major, N = B*H (head n = b*H + h)
 *   p    : caller-provided scratch of S doubles; receives the scores
 * Returns the index of the last visible key; *m_out receives m.
 */
static int64_t row_scores(const double* q, const double* k, double* p, int64_t S, int64_t d, int causal,
                          double scale, int64_t n, int64_t i, double* m_out) {
  const double* qi = q + (n * S + i) * d;
  const double* kh = k + n * S * d;
  int64_t last = causal ? i : S - 1; /* last visible key */
  for (int64_t j = 0; j <= last; ++j) {
    double dot = 0.0;
    for (int64_t c = 0; c < d; ++c) dot += qi[c] * kh[j * d + c];
    p[j] = scale * dot;
  }
  double m = p[0];
  for (int64_t j = 1; j <= last; ++j)
    if (p[j] > m) m = p[j];
  *m_out = m;
  return last;
}

/*
 * One query row of one head, steps 4-5 after row_scores:
 *   4. p_j = exp(s_j - m), l = sum_j p_j
 *   5. o[c] = (sum_j p_j * v[n,j,c]) / l
 */
static void attn_one_row(const double* q, const double* k, const double* v,
                         double* o_row, double* p, int64_t S, int64_t d,
                         int causal, double scale, int64_t n, int64_t i) {
  const double* vh = v + n * S * d;
  double m;
  int64_t last = row_scores(q, k, p, S, d, causal, scale, n, i, &m);
  /* 4. unnormalised probabilities and their sum */
  double l = 0.0;
  for (int64_t j = 0; j <= last; ++j) {
    p[j] = exp(p[j] - m);
    l += p[j];
  }
  /* 5. weighted sum of the value rows, divided by the sum */
  for (int64_t c = 0; c < d; ++c) {
    double acc = 0.0;
    for (int64_t j = 0; j <= last; ++j) acc += p[j] * vh[j * d + c];
    o_row[c] = acc / l;
  }
}

static int attn_args_ok(const void* q, const void* k, const void* v, const void* o,
                        int64_t S, int64_t d, double scale) {
  if (!q || !k || !v || !o) return 0;
  if (S < 1 || d < 1) return 0;
  if (!(scale == scale) || isinf(scale)) return 0;
  return 1;
}

/* Full attention forward: o[n,i,:] for every head n < B*H and query i < S. */
int kb_oracle_attn(const double* q, const double* k, const double* v, double* o,
                   int64_t B, int64_t H, int64_t S, int64_t d, int causal,
                   double scale) {
  if (B < 1 || H < 1 || !attn_args_ok(q, k, v, o, S, d, scale)) return KB_ORACLE_BAD_ARG;
  double* p = (double*)malloc((size_t)S * sizeof(double));
  if (!p) return KB_ORACLE_NO_MEMORY;
  int64_t N = B * H;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t i = 0; i < S; ++i)
      attn_one_row(q, k, v, o + (n * S + i) * d, p, S, d, causal, scale, n, i);
  free(p);
  return KB_ORACLE_OK;
}

/*
 * Log-sum-exp of every score row: lse[n,i] = log(sum_j exp(s_j)) over the
 * visible keys (the natural log of the softmax denominator; the flash page's
 * running max m and denominator l give it as m + log l). Computed as
 * m + log(sum_j exp(s_j - m)) with the row maximum m. lse is [N, S].
 */
int kb_oracle_lse(const double* q, const double* k, double* lse, int64_t N, int64_t S, int64_t d,
                  int causal, double scale) {
  if (N < 1 || !lse || !attn_args_ok(q, k, k, lse, S, d, scale)) return KB_ORACLE_BAD_ARG;
  double* p = (double*)malloc((size_t)S * sizeof(double));
  if (!p) return KB_ORACLE_NO_MEMORY;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t i = 0; i < S; ++i) {
      double m;
      int64_t last = row_scores(q, k, p, S, d, causal, scale, n, i, &m);
      double l = 0.0;
      for (int64_t j = 0; j <= last; ++j) l += exp(p[j] - m);
      lse[n * S + i] = m + log(l);
    }
  }
  free(p);
  return KB_ORACLE_OK;
}

/*
 * A listed subset of (head, query) rows, for workloads too large to evaluate
 * in full. Rows are independent, so each listed row is exactly the row the
 * full evaluation would give. o is [count, d].
 */
int kb_oracle_attn_rows(const double* q, const double* k, const double* v, double* o,
                        int64_t N, int64_t S, int64_t d, int causal, double scale,
                        const int64_t* heads, const int64_t* rows, int64_t count) {
  if (N < 1 || count < 0 || !attn_args_ok(q, k, v, o, S, d, scale)) return KB_ORACLE_BAD_ARG;
  if (count > 0 && (!heads || !rows)) return KB_ORACLE_BAD_ARG;
  for (int64_t t = 0; t < count; ++t)
    if (heads[t] < 0 || heads[t] >= N || rows[t] < 0 || rows[t] >= S) return KB_ORACLE_BAD_ARG;
  double* p = (double*)malloc((size_t)S * sizeof(double));
  if (!p) return KB_ORACLE_NO_MEMORY;
  for (int64_t t = 0; t < count; ++t)
    attn_one_row(q, k, v, o + t * d, p, S, d, causal, scale, heads[t], rows[t]);
  free(p);
  return KB_ORACLE_OK;
}

/*
 * The Triad's sibling reference kernels (TileOPs README, "HBM Bandwidth" /
 * "Methodology": copy 1:1 read:write, read-only, write-only):
 *   copy : a[i] = b[i]
 *   fill : a[i] = s             (write-only)
 *   sum  : sum_i b[i] in double (read-only; the value a reader must produce)
 */
int kb_oracle_copy(float* a, const float* b, int64_t n) {
  if (n < 0 || (n > 0 && (!a || !b))) return KB_ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) a[i] = b[i];
  return KB_ORACLE_OK;
}

int kb_oracle_fill(float* a, float s, int64_t n) {
  if (n < 0 || (n > 0 && !a)) return KB_ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) a[i] = s;
  return KB_ORACLE_OK;
}

int kb_oracle_sum(const float* b, int64_t n, double* out) {
  if (n < 0 || !out || (n > 0 && !b)) return KB_ORACLE_BAD_ARG;
  double acc = 0.0;
  for (int64_t i = 0; i < n; ++i) acc += (double)b[i];
  *out = acc;
  return KB_ORACLE_OK;
}

/*
 * STREAM Triad, a[i] = b[i] + s*c[i], in fp32 with one rounding of the exact
 * value (C99 fmaf is specified to round b + s*c once).
 */
int kb_oracle_triad(float* a, const float* b, const float* c, float s, int64_t n) {
  if (n < 0 || (n > 0 && (!a || !b || !c))) return KB_ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) a[i] = fmaf(s, c[i], b[i]);
  return KB_ORACLE_OK;
}

/* --------------------------------------------------------------------------
 * Q15 fixed-point model of the microcontroller path.
 *
 * kbench page, section "CPU reference + cache profiling": the second CPU
 * reference is a bit-accurate model of the board's fixed-point path, with Q15
 * inputs, Q15.16 score accumulation and a 64-entry exp table. Section
 * "ARM Cortex-M4 firmware": that path handles one query row at a time and
 * streams the keys like the flash kernel, with an online-rescaled softmax, in
 * scalar fixed point because the core has no hardware exp.
 *
 * The pages print neither the table nor any rounding rule. The readings taken
 * here (the plainest fixed-point choices):
 *   Q15      int16, value = x / 2^15.
 *   Q15.16   int64 holding value * 2^16 (scores, in base-2 units).
 *   score    the exact integer sum of the d products q_c * k_c (Q30), shifted
 *            right by 14 (floor) to Q15.16, then multiplied by
 *            C = round(scale * log2(e) * 2^16) and shifted right by 16
 *            (floor), so that exp(x) becomes 2^z.
 *   exp      2^(-t) for t >= 0 in Q15.16 is T[f] >> n, where n = floor(t),
 *            f = the top 6 bits of the fraction of t, and the 64-entry table
 *            holds T[f] = round(2^15 * 2^(-f/64)); the result is 0 once
 *            n >= 16. Weights p are therefore Q15 in [0, 2^15].
 *   stream   keys in tiles of 32 from key 0 (the last tile clipped to the
 *            last visible key). For each tile: its scores and their maximum;
 *            if the maximum rose above the running maximum m, scale l and
 *            every acc_c by a = 2^(-(m_new - m)) (product shifted right by
 *            15, floor) and set m = m_new; then for each key p = 2^(-(m - z)),
 *            l += p, acc_c += p * v_c (exact, Q30).
 *   output   o_c = acc_c / l rounded to nearest (halves away from zero),
 *            saturated to int16.
 * Limits that keep every intermediate inside int64: S <= 65536, d <= 1024,
 * C <= 2^30.
 * -------------------------------------------------------------------------- */
#define KB_Q15_TILE 32
#define KB_Q15_LOG2E 1.4426950408889634074

/* floor(x / 2^s), written without relying on how >> treats negative values */
static int64_t q15_floor_shift(int64_t x, int s) {
  const int64_t p = (int64_t)1 << s;
  return x >= 0 ? x / p : -((-x + p - 1) / p);
}

/* T[f] = round(2^15 * 2^(-f/64)), f = 0..63 */
static void q15_exp_table(uint16_t t[64]) {
  for (int f = 0; f < 64; ++f) t[f] = (uint16_t)llround(32768.0 * exp2(-(double)f / 64.0));
}

/* 2^(-t) in Q15 for t >= 0 in Q15.16, from the table */
static int64_t q15_pow2_neg(int64_t t, const uint16_t tab[64]) {
  const int64_t n = t / 65536;          /* integer part */
  const int64_t f = (t % 65536) / 1024; /* top 6 bits of the fraction */
  if (n >= 16) return 0;
  return (int64_t)tab[f] / ((int64_t)1 << n);
}

/* a / b for b > 0, rounded to nearest with halves away from zero */
static int64_t q15_round_div(int64_t a, int64_t b) {
  return a >= 0 ? (a + b / 2) / b : -((-a + b / 2) / b);
}

/* One query row of one head; acc is scratch of d int64. */
static void q15_one_row(const int16_t* q, const int16_t* k, const int16_t* v, int16_t* o_row,
                        int64_t* acc, int64_t S, int64_t d, int causal, int64_t C,
                        const uint16_t tab[64], int64_t n, int64_t i) {
  const int16_t* qi = q + (n * S + i) * d;
  const int16_t* kh = k + n * S * d;
  const int16_t* vh = v + n * S * d;
  const int64_t last_key = causal ? i : S - 1;
  int64_t z[KB_Q15_TILE];
  int64_t m = 0, l = 0;
  int have_m = 0;
  for (int64_t c = 0; c < d; ++c) acc[c] = 0;
  for (int64_t t0 = 0; t0 <= last_key; t0 += KB_Q15_TILE) {
    const int64_t t1 = t0 + KB_Q15_TILE - 1 < last_key ? t0 + KB_Q15_TILE - 1 : last_key;
    /* scores of the tile (Q15.16, base 2) and the tile maximum */
    int64_t mt = 0;
    for (int64_t j = t0; j <= t1; ++j) {
      int64_t dot = 0;
      for (int64_t c = 0; c < d; ++c) dot += (int64_t)qi[c] * (int64_t)kh[j * d + c];
      const int64_t s16 = q15_floor_shift(dot, 14);
      z[j - t0] = q15_floor_shift(s16 * C, 16);
      if (j == t0 || z[j - t0] > mt) mt = z[j - t0];
    }
    /* online rescale when the running maximum rises */
    if (!have_m) {
      m = mt;
      have_m = 1;
    } else if (mt > m) {
      const int64_t a = q15_pow2_neg(mt - m, tab);
      l = q15_floor_shift(l * a, 15);
      for (int64_t c = 0; c < d; ++c) acc[c] = q15_floor_shift(acc[c] * a, 15);
      m = mt;
    }
    /* weights of the tile's keys, accumulated */
    for (int64_t j = t0; j <= t1; ++j) {
      const int64_t p = q15_pow2_neg(m - z[j - t0], tab);
      l += p;
      for (int64_t c = 0; c < d; ++c) acc[c] += p * (int64_t)vh[j * d + c];
    }
  }
  for (int64_t c = 0; c < d; ++c) {
    int64_t r = q15_round_div(acc[c], l);
    if (r > 32767) r = 32767;
    if (r < -32768) r = -32768;
    o_row[c] = (int16_t)r;
  }
}

/* The 64-entry exp table of the Q15 model. */
int kb_oracle_q15_exp_table(uint16_t* out) {
  if (!out) return KB_ORACLE_BAD_ARG;
  q15_exp_table(out);
  return KB_ORACLE_OK;
}

/* Q15 attention forward over [N, S, d] int16 tensors (head n = b*H + h). */
int kb_oracle_attn_q15(const int16_t* q, const int16_t* k, const int16_t* v, int16_t* o,
                       int64_t N, int64_t S, int64_t d, int causal, double scale) {
  if (!q || !k || !v || !o || N < 1 || S < 1 || S > 65536 || d < 1 || d > 1024) return KB_ORACLE_BAD_ARG;
  if (!(scale > 0.0) || isinf(scale)) return KB_ORACLE_BAD_ARG;
  const double cd = scale * KB_Q15_LOG2E * 65536.0;
  if (!(cd <= 1073741824.0)) return KB_ORACLE_BAD_ARG;
  const int64_t C = llround(cd);
  uint16_t tab[64];
  q15_exp_table(tab);
  int64_t* acc = (int64_t*)malloc((size_t)d * sizeof(int64_t));
  if (!acc) return KB_ORACLE_NO_MEMORY;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t i = 0; i < S; ++i) q15_one_row(q, k, v, o + (n * S + i) * d, acc, S, d, causal, C, tab, n, i);
  free(acc);
  return KB_ORACLE_OK;
}
