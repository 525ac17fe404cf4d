/*
 * gdr_oracle.c -- fp64 CPU oracle for the gated delta rule, forward and backward.
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

/*
 * Backward of the recurrence above (reverse-mode differentiation, token by token).
 *
 * The pages describe a training backend whose backward is bit-reproducible and
 * tolerates length-0 segments ("Findings ...", intro and section 2) but print no
 * backward formula; this is the gradient of the forward defined above.  Given
 * dL/do_t (`dout`) and dL/dht (`dht`, or zero), with D the total gradient of the
 * loss with respect to the state after token t (starting from dht at the last
 * token), x = S_{t-1}^T k, y = D^T k, a = exp(g_t), b = beta_t, for t from the
 * last token of a segment down to the first:
 *
 *     D    += scale q_t do_t^T               (o_t = scale S_t^T q_t)
 *     dq_t  = scale S_t do_t
 *     dv_t  = b y
 *     dbeta_t = y . (v_t - a x)
 *     dk_t  = b D (v_t - a x) - a b S_{t-1} y
 *     dg_t  = a (<D, S_{t-1}> - b y . x)
 *     D    <- a (D - b k_t y^T)              (the gradient for S_{t-1})
 *
 * and dh0 = D after the first token.  These follow from the delta form
 * S_t = a S_{t-1} + k u^T, u = b (v - a S_{t-1}^T k), by the chain rule.
 *
 * States S_{t-1}, S_t are needed in reverse order: the forward keeps the state
 * at the start of every 64-token block of the segment and each block's states
 * are recomputed (with the same arithmetic) when the backward reaches it.
 *
 * Outputs (double, caller-zeroed): dq_h and dk_h are PER VALUE HEAD
 * [T, H, dk] (the caller sums the value heads of a query/key head);
 * dv [T, H, dv]; dg, dbeta [T, H]; dh0 [n_seq, H, dk, dv] or NULL.
 */
enum { ORC_BLK = 64 };

/* exp of a stored gate value (the backward's decay factor a = e^g) */
static double orc_gate(const void *g, int g_dt, int64_t i) { return exp(orc_load(g, g_dt, i)); }

/* One token of the forward in the delta form: S <- a S + k u^T, u = b (v - a S^T k). */
static void orc_step(double *S, const double *kv, const double *vv, double a, double b,
                     double *x, double *u, int32_t dk, int32_t dv) {
  for (int32_t j = 0; j < dv; ++j) x[j] = 0.0;
  for (int32_t i = 0; i < dk; ++i)
    for (int32_t j = 0; j < dv; ++j) x[j] += S[(int64_t)i * dv + j] * kv[i];
  for (int32_t j = 0; j < dv; ++j) u[j] = (vv[j] - a * x[j]) * b;
  for (int32_t i = 0; i < dk; ++i)
    for (int32_t j = 0; j < dv; ++j)
      S[(int64_t)i * dv + j] = a * S[(int64_t)i * dv + j] + kv[i] * u[j];
}

int gdr_oracle_recurrent_bwd(const void *q, int q_dt, const void *k, int k_dt,
                             const void *v, int v_dt, const void *g, int g_dt,
                             const void *beta, int beta_dt, double scale,
                             const void *h0, int h0_dt, const int32_t *cu_seqlens,
                             int32_t n_seq, int64_t T, int32_t Hk, int32_t H,
                             int32_t dk, int32_t dv, const void *dout, int do_dt,
                             const void *dht, int dht_dt, double *dq_h, double *dk_h,
                             double *dv_out, double *dg, double *dbeta, double *dh0,
                             int n_threads) {
  if (!q || !k || !v || !g || !beta || !cu_seqlens || !dout) return -1;
  if (!dq_h || !dk_h || !dv_out || !dg || !dbeta) return -1;
  if (n_seq < 0 || T < 0 || Hk <= 0 || H <= 0 || dk <= 0 || dv <= 0) return -2;
  if (H % Hk != 0) return -3;
  const int32_t group = H / Hk;
  const int64_t units = (int64_t)n_seq * H;
  const int64_t SS = (int64_t)dk * dv;
  int bad = 0;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double *D = (double *)malloc(sizeof(double) * (size_t)SS);
    double *blk = (double *)malloc(sizeof(double) * (size_t)SS * (ORC_BLK + 1));
    double *x = (double *)malloc(sizeof(double) * (size_t)dv);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    double *y = (double *)malloc(sizeof(double) * (size_t)dv);
    double *w = (double *)malloc(sizeof(double) * (size_t)dv);
    double *kv = (double *)malloc(sizeof(double) * (size_t)dk);
    double *qv = (double *)malloc(sizeof(double) * (size_t)dk);
    double *vv = (double *)malloc(sizeof(double) * (size_t)dv);
    double *dov = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!D || !blk || !x || !u || !y || !w || !kv || !qv || !vv || !dov) {
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
        const int32_t hq = h / group;
        int64_t s, e;
        orc_bounds(cu_seqlens, n, T, &s, &e);
        const int64_t len = e - s, nblk = (len + ORC_BLK - 1) / ORC_BLK;
        /* states at the start of every block */
        double *starts = (double *)malloc(sizeof(double) * (size_t)SS * (size_t)(nblk > 0 ? nblk : 1));
        if (!starts) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
          bad = 1;
          continue;
        }
        for (int64_t i = 0; i < SS; ++i)
          blk[i] = h0 ? orc_load(h0, h0_dt, ((int64_t)n * H + h) * SS + i) : 0.0;
        for (int64_t tf = s; tf < e; ++tf) {
          const int64_t t = tf;
          if ((t - s) % ORC_BLK == 0) memcpy(starts + ((t - s) / ORC_BLK) * SS, blk, sizeof(double) * (size_t)SS);
          const double a = orc_gate(g, g_dt, t * H + h);
          const double b = orc_load(beta, beta_dt, t * H + h);
          for (int32_t i = 0; i < dk; ++i) kv[i] = orc_load(k, k_dt, (t * Hk + hq) * (int64_t)dk + i);
          for (int32_t j = 0; j < dv; ++j) vv[j] = orc_load(v, v_dt, (t * H + h) * (int64_t)dv + j);
          orc_step(blk, kv, vv, a, b, x, u, dk, dv);
        }
        /* D = dL/dS after the last token */
        for (int64_t i = 0; i < SS; ++i)
          D[i] = dht ? orc_load(dht, dht_dt, ((int64_t)n * H + h) * SS + i) : 0.0;
        for (int64_t bi = nblk - 1; bi >= 0; --bi) {
          const int64_t tb = s + bi * ORC_BLK, te = (tb + ORC_BLK < e) ? tb + ORC_BLK : e;
          /* blk[r] = state before token tb + r, r = 0 .. te - tb */
          memcpy(blk, starts + bi * SS, sizeof(double) * (size_t)SS);
          for (int64_t t = tb; t < te; ++t) {
            double *next = blk + (t - tb + 1) * SS;
            memcpy(next, blk + (t - tb) * SS, sizeof(double) * (size_t)SS);
            const double a = orc_gate(g, g_dt, t * H + h);
            const double b = orc_load(beta, beta_dt, t * H + h);
            for (int32_t i = 0; i < dk; ++i) kv[i] = orc_load(k, k_dt, (t * Hk + hq) * (int64_t)dk + i);
            for (int32_t j = 0; j < dv; ++j) vv[j] = orc_load(v, v_dt, (t * H + h) * (int64_t)dv + j);
            orc_step(next, kv, vv, a, b, x, u, dk, dv);
          }
          for (int64_t t = te - 1; t >= tb; --t) {
            const double *Sp = blk + (t - tb) * SS;     /* S_{t-1} */
            const double *St = blk + (t - tb + 1) * SS; /* S_t */
            const double a = orc_gate(g, g_dt, t * H + h);
            const double b = orc_load(beta, beta_dt, t * H + h);
            const int64_t qk_base = (t * Hk + hq) * (int64_t)dk, v_base = (t * H + h) * (int64_t)dv;
            for (int32_t i = 0; i < dk; ++i) {
              kv[i] = orc_load(k, k_dt, qk_base + i);
              qv[i] = orc_load(q, q_dt, qk_base + i);
            }
            for (int32_t j = 0; j < dv; ++j) {
              vv[j] = orc_load(v, v_dt, v_base + j);
              dov[j] = orc_load(dout, do_dt, v_base + j);
            }
            /* D += scale q do^T */
            for (int32_t i = 0; i < dk; ++i)
              for (int32_t j = 0; j < dv; ++j) D[(int64_t)i * dv + j] += scale * qv[i] * dov[j];
            /* dq_t = scale S_t do_t */
            double *dqt = dq_h + (t * H + h) * (int64_t)dk;
            for (int32_t i = 0; i < dk; ++i) {
              double acc = 0.0;
              for (int32_t j = 0; j < dv; ++j) acc += St[(int64_t)i * dv + j] * dov[j];
              dqt[i] = scale * acc;
            }
            /* x = S_{t-1}^T k, y = D^T k, w = v - a x */
            for (int32_t j = 0; j < dv; ++j) { x[j] = 0.0; y[j] = 0.0; }
            for (int32_t i = 0; i < dk; ++i)
              for (int32_t j = 0; j < dv; ++j) {
                x[j] += Sp[(int64_t)i * dv + j] * kv[i];
                y[j] += D[(int64_t)i * dv + j] * kv[i];
              }
            double yw = 0.0, yx = 0.0, dsp = 0.0;
            for (int32_t j = 0; j < dv; ++j) {
              w[j] = vv[j] - a * x[j];
              yw += y[j] * w[j];
              yx += y[j] * x[j];
            }
            for (int64_t i = 0; i < SS; ++i) dsp += D[i] * Sp[i];
            double *dvt = dv_out + v_base;
            for (int32_t j = 0; j < dv; ++j) dvt[j] = b * y[j];
            dbeta[t * H + h] = yw;
            dg[t * H + h] = a * (dsp - b * yx);
            /* dk_t = b D w - a b S_{t-1} y */
            double *dkt = dk_h + (t * H + h) * (int64_t)dk;
            for (int32_t i = 0; i < dk; ++i) {
              double dw = 0.0, sy = 0.0;
              for (int32_t j = 0; j < dv; ++j) {
                dw += D[(int64_t)i * dv + j] * w[j];
                sy += Sp[(int64_t)i * dv + j] * y[j];
              }
              dkt[i] = b * dw - a * b * sy;
            }
            /* D <- a (D - b k y^T) */
            for (int32_t i = 0; i < dk; ++i)
              for (int32_t j = 0; j < dv; ++j)
                D[(int64_t)i * dv + j] = a * (D[(int64_t)i * dv + j] - b * kv[i] * y[j]);
          }
        }
        if (dh0) memcpy(dh0 + ((int64_t)n * H + h) * SS, D, sizeof(double) * (size_t)SS);
        free(starts);
      }
    }
    free(D);
    free(blk);
    free(x);
    free(u);
    free(y);
    free(w);
    free(kv);
    free(qv);
    free(vv);
    free(dov);
  }
  return bad ? -4 : 0;
}

int gdr_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
