/*
 * gdr_oracle.c -- fp64 CPU oracle for the gated delta rule forward.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline leg load this file.  It shares no code, header or constant with
 * the CUDA path and is deliberately slow and plain.
 *
 * What it computes: the gated delta rule recurrence, token by token, in
 * double precision, for every (segment n, value head h):
 *
 *     S_0   = h0[n, h]            (or zero)
 *     S_t   = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t   = scale * S_t^T q_t
 *     ht[n, h] = S_last
 *
 * with S a dk x dv matrix stored row-major (row = key dimension).  The update
 * is evaluated in the algebraically identical delta form
 *
 *     x = S^T k;   u = beta (v - exp(g) x);   S <- exp(g) S + k u^T.
 *
 * This is the recurrence the FlashQLA GDN kernels evaluate ("Findings from
 * integrating FlashQLA's Blackwell GDN kernels into a JAX trainer", intro:
 * "Gated Delta Rule kernels"); the pages do not print the formula, so the
 * formula above is the operator's stated definition.
 *
 * Segments ("Findings ...", section 2): segment n covers tokens
 * [c[n], c[n+1]) where c is cu_seqlens made non-decreasing by a running
 * maximum and clamped to [0, T].  Empty segments write no output and, when ht
 * is requested, leave ht[n] = h0[n] (or zero).  Tokens outside every segment
 * are not written.
 *
 * Grouped heads: value head h reads query/key head h / (H / Hk).
 *
 * State checkpoints (gdr_oracle_recurrent_ckpt): every `ckpt_every` tokens of a
 * segment the state is copied out, as for prefix caching ("feat(cake_kda): add
 * paired recurrent training for SM100a and SM103a", the released inference
 * surface keeps state checkpoints every N tokens).  Checkpoint m (m = 1, 2, ...,
 * floor(len / ckpt_every)) of segment n is S after the segment's first
 * m * ckpt_every tokens; segment n's checkpoints fill rows ckpt_off[n] ..
 * ckpt_off[n + 1] - 1 of ckpt[rows, H, dk, dv], ckpt_off being the running sum
 * of floor(len / ckpt_every).
 *
 * Inputs are read in their stored precision (bf16 bits, fp32 or fp64) and
 * promoted exactly to double.  Outputs are double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

static double orc_load(const void *p, int dt, int64_t i) {
  if (dt == ORC_F64) return ((const double *)p)[i];
  if (dt == ORC_F32) return (double)((const float *)p)[i];
  /* bf16: the upper 16 bits of an IEEE binary32 */
  uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Segment bounds after the running-maximum / clamp reading of cu_seqlens. */
static void orc_bounds(const int32_t *cu, int32_t n, int64_t T, int64_t *s, int64_t *e) {
  int64_t lo = 0, prev = 0;
  for (int32_t i = 0; i <= n + 1; ++i) {
    int64_t c = cu[i];
    if (c < 0) c = 0;
    if (c > T) c = T;
    if (i > 0 && c < prev) c = prev;
    if (i == n) lo = c;
    prev = c;
  }
  *s = lo;
  *e = prev;
}

static int orc_run(const void *q, int q_dt, const void *k, int k_dt,
                   const void *v, int v_dt, const void *g, int g_dt,
                   const void *beta, int beta_dt, double scale,
                   const void *h0, int h0_dt, const int32_t *cu_seqlens,
                   int32_t n_seq, int64_t T, int32_t Hk, int32_t H,
                   int32_t dk, int32_t dv, double *o, double *ht,
                   int32_t ckpt_every, double *ckpt, const int32_t *ckpt_off,
                   int n_threads) {
  if (!q || !k || !v || !g || !beta || !cu_seqlens || !o) return -1;
  if (n_seq < 0 || T < 0 || Hk <= 0 || H <= 0 || dk <= 0 || dv <= 0) return -2;
  if (H % Hk != 0) return -3;
  const int32_t group = H / Hk;
  const int64_t units = (int64_t)n_seq * H;
  int bad = 0;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *x = (double *)malloc(sizeof(double) * (size_t)dv);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    double *kv = (double *)malloc(sizeof(double) * (size_t)dk);
    double *qv = (double *)malloc(sizeof(double) * (size_t)dk);
    if (!S || !x || !u || !kv || !qv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      bad = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t unit = 0; unit < units; ++unit) {
        const int32_t n = (int32_t)(unit / H);
        const int32_t h = (int32_t)(unit % H);
        const int32_t hk = h / group;
        int64_t s, e;
        orc_bounds(cu_seqlens, n, T, &s, &e);
        for (int64_t i = 0; i < (int64_t)dk * dv; ++i)
          S[i] = h0 ? orc_load(h0, h0_dt, ((int64_t)n * H + h) * dk * dv + i) : 0.0;
        for (int64_t t = s; t < e; ++t) {
          const double alpha = exp(orc_load(g, g_dt, t * H + h));
          const double b = orc_load(beta, beta_dt, t * H + h);
          const int64_t qk_base = (t * Hk + hk) * (int64_t)dk;
          const int64_t v_base = (t * H + h) * (int64_t)dv;
          for (int32_t i = 0; i < dk; ++i) {
            kv[i] = orc_load(k, k_dt, qk_base + i);
            qv[i] = orc_load(q, q_dt, qk_base + i);
          }
          /* x = S^T k */
          for (int32_t j = 0; j < dv; ++j) x[j] = 0.0;
          for (int32_t i = 0; i < dk; ++i) {
            const double ki = kv[i];
            const double *row = S + (int64_t)i * dv;
            for (int32_t j = 0; j < dv; ++j) x[j] += row[j] * ki;
          }
          /* u = beta (v - alpha x) */
          for (int32_t j = 0; j < dv; ++j)
            u[j] = b * (orc_load(v, v_dt, v_base + j) - alpha * x[j]);
          /* S <- alpha S + k u^T */
          for (int32_t i = 0; i < dk; ++i) {
            const double ki = kv[i];
            double *row = S + (int64_t)i * dv;
            for (int32_t j = 0; j < dv; ++j) row[j] = alpha * row[j] + ki * u[j];
          }
          /* o_t = scale S^T q */
          double *ot = o + v_base;
          for (int32_t j = 0; j < dv; ++j) ot[j] = 0.0;
          for (int32_t i = 0; i < dk; ++i) {
            const double qi = qv[i];
            const double *row = S + (int64_t)i * dv;
            for (int32_t j = 0; j < dv; ++j) ot[j] += row[j] * qi;
          }
          for (int32_t j = 0; j < dv; ++j) ot[j] *= scale;
          /* state checkpoint after the segment's first m * ckpt_every tokens */
          if (ckpt && (t - s + 1) % ckpt_every == 0) {
            const int64_t row = ckpt_off[n] + (t - s + 1) / ckpt_every - 1;
            memcpy(ckpt + (row * H + h) * dk * dv, S, sizeof(double) * (size_t)dk * dv);
          }
        }
        if (ht) memcpy(ht + ((int64_t)n * H + h) * dk * dv, S, sizeof(double) * (size_t)dk * dv);
      }
    }
    free(S);
    free(x);
    free(u);
    free(kv);
    free(qv);
  }
  return bad ? -4 : 0;
}

int gdr_oracle_recurrent(const void *q, int q_dt, const void *k, int k_dt,
                         const void *v, int v_dt, const void *g, int g_dt,
                         const void *beta, int beta_dt, double scale,
                         const void *h0, int h0_dt, const int32_t *cu_seqlens,
                         int32_t n_seq, int64_t T, int32_t Hk, int32_t H,
                         int32_t dk, int32_t dv, double *o, double *ht,
                         int n_threads) {
  return orc_run(q, q_dt, k, k_dt, v, v_dt, g, g_dt, beta, beta_dt, scale, h0, h0_dt,
                 cu_seqlens, n_seq, T, Hk, H, dk, dv, o, ht, 0, NULL, NULL, n_threads);
}

/* As gdr_oracle_recurrent, plus state checkpoints (see the header comment).
 * ckpt_off [n_seq + 1] is written here; ckpt needs ckpt_off[n_seq] rows. */
int gdr_oracle_recurrent_ckpt(const void *q, int q_dt, const void *k, int k_dt,
                              const void *v, int v_dt, const void *g, int g_dt,
                              const void *beta, int beta_dt, double scale,
                              const void *h0, int h0_dt, const int32_t *cu_seqlens,
                              int32_t n_seq, int64_t T, int32_t Hk, int32_t H,
                              int32_t dk, int32_t dv, double *o, double *ht,
                              int32_t ckpt_every, double *ckpt, int32_t *ckpt_off,
                              int n_threads) {
  if (ckpt_every <= 0 || !ckpt || !ckpt_off || !cu_seqlens || n_seq < 0) return -5;
  ckpt_off[0] = 0;
  for (int32_t n = 0; n < n_seq; ++n) {
    int64_t s, e;
    orc_bounds(cu_seqlens, n, T, &s, &e);
    ckpt_off[n + 1] = ckpt_off[n] + (int32_t)((e - s) / ckpt_every);
  }
  return orc_run(q, q_dt, k, k_dt, v, v_dt, g, g_dt, beta, beta_dt, scale, h0, h0_dt,
                 cu_seqlens, n_seq, T, Hk, H, dk, dv, o, ht, ckpt_every, ckpt, ckpt_off,
                 n_threads);
}

int gdr_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
