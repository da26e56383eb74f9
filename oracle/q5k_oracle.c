/*
 * f64 CPU oracle of the Muse Glimmer decode output stage.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package entry's smoke check and the
 * benchmark's CPU-baseline / reference leg may load or call this file.  The
 * CUDA path never links, imports or reads it, and it shares no code, header,
 * table or constant with the CUDA path.
 *
 * What it computes, in the order "Chapter 20 — Final norm, LM head, and the
 * soft cap" gives (§20.1, and the CPU oracle tail quoted in §20.4):
 *   1. final RMSNorm (§20.1; "Chapter 9 — The Muse Glimmer architecture" §9.5):
 *        r = 1 / sqrt(sum_j h_j^2 / K + eps),  x_j = h_j * r * gamma_j
 *      (skipped when gamma is NULL: then x = h)
 *   2. LM-head matvec (§20.1): raw_i = sum_j W[i, j] * x_j, W stored as Q5_K
 *      super-blocks (§20.3: 256 weights per 176-byte block), dequantised by
 *      this file's own parser: W = d * sc_s * q - dmin * m_s
 *   3. logit scale, then soft cap (§20.1, §20.4; Chapter 9 §9.10):
 *        v = raw * scale;  out = cap > 0 ? cap * tanh(v / cap) : v
 * Everything is evaluated in binary64 with plain left-to-right sums; libm's
 * tanh, sqrt.  The greedy argmax (first index of the maximum) lives in the
 * Python side of the oracle.
 *
 * The Q5_K byte layout is not printed on the pages (they cite an absent
 * chapter for it).  The reading taken is ggml's block_q5_K: fp16 d, fp16 dmin,
 * 12 bytes of packed 6-bit scales and mins, 32 bytes of high bits, 128 bytes of
 * low nibbles.  Weight e of a block: sub-block s = e / 32, position l = e % 32;
 * low nibble = nibble (s & 1) of qs[32 * (s / 2) + l]; high bit = bit s of qh[l].
 * Scales: for s < 4, sc = scales[s] & 63 and m = scales[s + 4] & 63; for s >= 4,
 * sc = (scales[s + 4] & 15) | (scales[s - 4] >> 6) << 4 and
 * m = (scales[s + 4] >> 4) | (scales[s] >> 6) << 4.
 *
 * Q4_K (the FFN bulk's format, and the 756.5 MB alternative head of Chapter 20
 * §20.7: 144 bytes per 256 weights): the pages give only the block size.
 * Reading: ggml's block_q4_K — the same fp16 d, fp16 dmin and 12 scale bytes,
 * then 128 bytes of nibbles placed as in Q5_K, no high bits; q in 0..15 and
 * w = d * sc_s * q - dmin * m_s.
 *
 * Build: gcc -O2 -ffp-contract=off (no fused multiply-add, so every product and
 * sum is one correctly rounded binary64 operation, identical on x86 and Arm).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE binary16 bit pattern -> exact binary64 value (normals, subnormals, zero). */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 31;
  int mant = h & 1023;
  double v;
  if (ex == 0)
    v = ldexp((double)mant, -24);
  else if (ex == 31)
    v = mant ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + mant), ex - 25);
  return sign ? -v : v;
}

/* Parse one 176-byte block into its fields. */
void oracle_q5k_parse(const uint8_t *blk, double *d, double *dmin, int *sc, int *m,
                      int *q) {
  uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
  uint16_t mbits = (uint16_t)(blk[2] | (blk[3] << 8));
  *d = oracle_half_to_double(dbits);
  *dmin = oracle_half_to_double(mbits);
  const uint8_t *scales = blk + 4;
  const uint8_t *qh = blk + 16;
  const uint8_t *qs = blk + 48;
  for (int s = 0; s < 8; ++s) {
    if (s < 4) {
      sc[s] = scales[s] & 63;
      m[s] = scales[s + 4] & 63;
    } else {
      sc[s] = (scales[s + 4] & 15) | ((scales[s - 4] >> 6) << 4);
      m[s] = (scales[s + 4] >> 4) | ((scales[s] >> 6) << 4);
    }
  }
  for (int e = 0; e < 256; ++e) {
    int s = e / 32, l = e % 32;
    int lo = (qs[32 * (s / 2) + l] >> (4 * (s & 1))) & 15;
    int hi = (qh[l] >> s) & 1;
    q[e] = lo + 16 * hi;
  }
}

/* One Q4_K block: d, dmin, the eight 6-bit scales and mins, 256 quants 0..15. */
void oracle_q4k_parse(const uint8_t *blk, double *d, double *dmin, int *sc, int *m,
                      int *q) {
  *d = oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
  *dmin = oracle_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
  const uint8_t *scales = blk + 4;
  const uint8_t *qs = blk + 16;
  for (int s = 0; s < 8; ++s) {
    if (s < 4) {
      sc[s] = scales[s] & 63;
      m[s] = scales[s + 4] & 63;
    } else {
      sc[s] = (scales[s + 4] & 15) | ((scales[s - 4] >> 6) << 4);
      m[s] = (scales[s + 4] >> 4) | ((scales[s] >> 6) << 4);
    }
  }
  for (int e = 0; e < 256; ++e) {
    int s = e / 32, l = e % 32;
    q[e] = (qs[32 * (s / 2) + l] >> (4 * (s & 1))) & 15;
  }
}

/* The 256 weight values of one Q4_K block: w = d * sc_s * q - dmin * m_s. */
void oracle_q4k_dequant(const uint8_t *blk, double *w) {
  double d, dmin;
  int sc[8], m[8], q[256];
  oracle_q4k_parse(blk, &d, &dmin, sc, m, q);
  for (int e = 0; e < 256; ++e) {
    int s = e / 32;
    w[e] = d * (double)sc[s] * (double)q[e] - dmin * (double)m[s];
  }
}

/* The 256 weight values of one block: w = d * sc_s * q - dmin * m_s. */
void oracle_q5k_dequant(const uint8_t *blk, double *w) {
  double d, dmin;
  int sc[8], m[8], q[256];
  oracle_q5k_parse(blk, &d, &dmin, sc, m, q);
  for (int e = 0; e < 256; ++e) {
    int s = e / 32;
    w[e] = d * (double)sc[s] * (double)q[e] - dmin * (double)m[s];
  }
}

/* Final RMSNorm of one row, or the identity when gamma is NULL. */
void oracle_rmsnorm(const float *h, const float *gamma, int64_t k, double eps, double *x) {
  if (!gamma) {
    for (int64_t j = 0; j < k; ++j) x[j] = (double)h[j];
    return;
  }
  double ss = 0.0;
  for (int64_t j = 0; j < k; ++j) ss += (double)h[j] * (double)h[j];
  double r = 1.0 / sqrt(ss / (double)k + eps);
  for (int64_t j = 0; j < k; ++j) x[j] = (double)h[j] * r * (double)gamma[j];
}

/* Scale, then soft cap. */
double oracle_scale_softcap(double raw, double scale, double cap) {
  double v = raw * scale;
  return cap > 0.0 ? cap * tanh(v / cap) : v;
}

typedef struct {
  const double *x;       /* [batch][k] normed inputs */
  const uint8_t *w;      /* [n_rows][nb * block bytes] */
  int q4;                /* 1: Q4_K blocks (144 bytes), 0: Q5_K (176) */
  int64_t k, nb, batch, n_rows;
  double scale, cap;
  int64_t r0, r1;        /* output rows of this worker */
  const int64_t *rows;   /* optional explicit row list (length n_rows) */
  double *raw, *out;     /* [batch][n_rows] */
} lm_job;

static void *lm_worker(void *arg) {
  const lm_job *jb = (const lm_job *)arg;
  double *wrow = (double *)malloc(sizeof(double) * (size_t)jb->k);
  if (!wrow) return (void *)1;
  for (int64_t i = jb->r0; i < jb->r1; ++i) {
    int64_t row = jb->rows ? jb->rows[i] : i;
    const int64_t bb = jb->q4 ? 144 : 176;
    const uint8_t *src = jb->w + row * jb->nb * bb;
    for (int64_t kb = 0; kb < jb->nb; ++kb) {
      if (jb->q4) oracle_q4k_dequant(src + kb * bb, wrow + kb * 256);
      else oracle_q5k_dequant(src + kb * bb, wrow + kb * 256);
    }
    for (int64_t b = 0; b < jb->batch; ++b) {
      const double *xb = jb->x + b * jb->k;
      double acc = 0.0;
      for (int64_t j = 0; j < jb->k; ++j) acc += wrow[j] * xb[j];
      if (jb->raw) jb->raw[b * jb->n_rows + i] = acc;
      jb->out[b * jb->n_rows + i] = oracle_scale_softcap(acc, jb->scale, jb->cap);
    }
  }
  free(wrow);
  return NULL;
}

/*
 * The whole stage for `batch` hidden rows against an [n_w_rows x k] Q5_K
 * matrix.  If rows is NULL, every weight row 0..n_w_rows-1 is computed and
 * n_out = n_w_rows; otherwise the n_out listed weight rows are computed in that
 * order.  raw (optional) and out are [batch][n_out] binary64.
 * Returns 0, -1 on bad arguments, -2 on allocation failure.
 */
int oracle_lmhead_fmt(const float *hidden, int64_t batch, int64_t k, const float *gamma,
                      double eps, const uint8_t *w, int64_t n_w_rows, const int64_t *rows,
                      int64_t n_out, double scale, double cap, double *raw, double *out,
                      int nthreads, int q4) {
  if (!hidden || !w || !out || batch <= 0 || k <= 0 || k % 256) return -1;
  if (!rows) n_out = n_w_rows;
  if (n_out < 0) return -1;
  if (rows)
    for (int64_t i = 0; i < n_out; ++i)
      if (rows[i] < 0 || rows[i] >= n_w_rows) return -1;
  double *x = (double *)malloc(sizeof(double) * (size_t)(batch * k));
  if (!x) return -2;
  for (int64_t b = 0; b < batch; ++b) oracle_rmsnorm(hidden + b * k, gamma, k, eps, x + b * k);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n_out < 4 * nthreads) nthreads = 1;
  lm_job jobs[256];
  pthread_t th[256];
  unsigned char started[256];
  int rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    lm_job *jb = &jobs[t];
    jb->x = x; jb->w = w; jb->k = k; jb->nb = k / 256; jb->batch = batch;
    jb->n_rows = n_out; jb->scale = scale; jb->cap = cap; jb->rows = rows;
    jb->r0 = n_out * t / nthreads; jb->r1 = n_out * (t + 1) / nthreads;
    jb->raw = raw; jb->out = out;
    jb->q4 = q4;
  }
  for (int t = 0; t < nthreads; ++t) {
    started[t] = nthreads > 1 && pthread_create(&th[t], NULL, lm_worker, &jobs[t]) == 0;
    if (!started[t] && lm_worker(&jobs[t]) != NULL) rc = -2;
  }
  for (int t = 0; t < nthreads; ++t) {
    void *ret = NULL;
    if (started[t]) {
      pthread_join(th[t], &ret);
      if (ret != NULL) rc = -2;
    }
  }
  free(x);
  return rc;
}

/* The Q5_K stage (the LM head's format). */
int oracle_lmhead(const float *hidden, int64_t batch, int64_t k, const float *gamma,
                  double eps, const uint8_t *w, int64_t n_w_rows, const int64_t *rows,
                  int64_t n_out, double scale, double cap, double *raw, double *out,
                  int nthreads) {
  return oracle_lmhead_fmt(hidden, batch, k, gamma, eps, w, n_w_rows, rows, n_out, scale, cap,
                           raw, out, nthreads, 0);
}
