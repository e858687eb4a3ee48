/*
 * glinattn_oracle.c -- plain, slow, fp64 CPU oracle for the state-passing
 * linear-attention layer (gated linear attention and Gated DeltaNet).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load this library. The CUDA product path never links, loads
 * or calls it, and it shares no code, header or constant with that path.
 *
 * Every function is the plain definition, token by token, in double precision
 * (the front end has a single-precision twin, oracle_causal_conv_f32 and
 * oracle_l2norm_rows_f32, for bf16 activations, whose rounding to bf16 is a
 * decision taken in the precision the layer computes its front end in):
 *
 *   "Inference for linear attention and hybrid architectures",
 *   section "Two ways to write the same computation":
 *     - gated linear attention:  S_t = alpha_t S_{t-1} + k_t^T v_t,  o_t = q_t S_t
 *       (the output reads the state after the update, as the page's recurrent
 *       form does);
 *     - DeltaNet erases the old memory along k_t and then writes the new one,
 *       S_t = (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t, and Gated
 *       DeltaNet multiplies a decay gate alpha_t in.  Reading adopted for where
 *       the gate enters: S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1}
 *       + beta_t k_t^T v_t (the write term is not decayed), o_t = q_t S_t;
 *     - the short causal convolution (window about 4) in front of the layer,
 *       which keeps the last inputs of each request as part of the layer's
 *       cache.  Reading adopted: depthwise, width 4, tap 3 multiplies the
 *       current token, no bias, no activation, zero history for a fresh
 *       sequence; the cache holds the last 3 raw inputs, oldest first.
 *   section "Speculative decoding and PD disaggregation": one state is kept
 *   per draft position; a decode step reads and writes its request's state in
 *   a pool by slot index.
 *
 * Layouts (all row-major, innermost last):
 *   q, k    [B, T, H, dk]      v, o  [B, T, H, dv]
 *   alpha, beta [B, T, H]      S     [B, H, dk, dv]
 *   conv input x / output y [B, T, Cch], conv weight w [Cch, 4],
 *   conv cache [B, 3, Cch] (slot j holds x_{T-3+j}).
 *
 * Precondition checks return a negative code; nothing is clamped.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EBADARG (-1)
#define ORACLE_EGATE (-2) /* alpha outside (0, 1] or not finite */
#define ORACLE_ENOMEM (-3)

/* ------------------------------------------------------------------------ */
/* One (batch, head) sequence of the recurrence.                              */
/* ------------------------------------------------------------------------ */

typedef struct {
  int variant; /* 0 = gated linear attention, 1 = Gated DeltaNet */
  int B, T, H, dk, dv;
  const double *q, *k, *v, *alpha, *beta;
  double *S, *o, *states; /* states may be NULL */
  int status;
} recur_job;

static int recur_one(const recur_job *J, int b, int h, double *kS) {
  const int T = J->T, H = J->H, dk = J->dk, dv = J->dv;
  double *S = J->S + ((size_t)b * H + h) * dk * dv;
  for (int t = 0; t < T; ++t) {
    const size_t row = ((size_t)b * T + t) * H + h; /* index of (b, t, h) */
    const double *qt = J->q + row * dk;
    const double *kt = J->k + row * dk;
    const double *vt = J->v + row * dv;
    const double a = J->alpha[row];
    if (!(a > 0.0 && a <= 1.0)) return ORACLE_EGATE;

    if (J->variant == 0) {
      /* S = alpha S + k^T v */
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[i * dv + j] = a * S[i * dv + j] + kt[i] * vt[j];
    } else {
      /* S = alpha (I - beta k^T k) S + beta k^T v, applied as
         S' = alpha S;  S = S' - beta k^T (k S') + beta k^T v */
      const double bt = J->beta[row];
      for (int i = 0; i < dk * dv; ++i) S[i] *= a;
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += kt[i] * S[i * dv + j];
        kS[j] = acc;
      }
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
          S[i * dv + j] = S[i * dv + j] - bt * kt[i] * kS[j] + bt * kt[i] * vt[j];
    }

    /* o_t = q_t S_t (state after the update) */
    double *ot = J->o + row * dv;
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += qt[i] * S[i * dv + j];
      ot[j] = acc;
    }
    if (J->states) {
      double *dst = J->states + (((size_t)b * T + t) * H + h) * dk * dv;
      memcpy(dst, S, sizeof(double) * dk * dv);
    }
  }
  return ORACLE_OK;
}

typedef struct {
  recur_job *job;
  int first, last; /* unit range [first, last) over b * H + h */
} recur_task;

static void *recur_worker(void *arg) {
  recur_task *task = (recur_task *)arg;
  recur_job *J = task->job;
  double *kS = (double *)malloc(sizeof(double) * (J->dv > 0 ? J->dv : 1));
  int st = kS ? ORACLE_OK : ORACLE_ENOMEM;
  for (int u = task->first; u < task->last && st == ORACLE_OK; ++u)
    st = recur_one(J, u / J->H, u % J->H, kS);
  free(kS);
  if (st != ORACLE_OK) J->status = st; /* any failure is reported */
  return NULL;
}

/*
 * oracle_recurrence -- run the recurrence over T tokens for every (b, h).
 *   S (in/out) holds the start state on entry and the final state on exit.
 *   states (nullable) receives the state after every token, [B, T, H, dk, dv].
 *   nthreads <= 1 runs on the calling thread; otherwise (b, h) units are split
 *   statically over that many threads.  Returns 0 or a negative code.
 */
int oracle_recurrence(int variant, int B, int T, int H, int dk, int dv, const double *q,
                      const double *k, const double *v, const double *alpha, const double *beta,
                      double *S, double *o, double *states, int nthreads) {
  if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return ORACLE_EBADARG;
  if (variant != 0 && variant != 1) return ORACLE_EBADARG;
  if (variant == 1 && !beta) return ORACLE_EBADARG;
  recur_job J = {variant, B, T, H, dk, dv, q, k, v, alpha, beta, S, o, states, ORACLE_OK};
  const int units = B * H;
  if (units == 0 || T == 0) return ORACLE_OK;
  if (nthreads > units) nthreads = units;
  if (nthreads <= 1) {
    recur_task task = {&J, 0, units};
    recur_worker(&task);
    return J.status;
  }
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
  recur_task *tasks = (recur_task *)malloc(sizeof(recur_task) * nthreads);
  if (!tid || !tasks) {
    free(tid);
    free(tasks);
    return ORACLE_ENOMEM;
  }
  for (int i = 0; i < nthreads; ++i) {
    tasks[i].job = &J;
    tasks[i].first = (int)((long long)units * i / nthreads);
    tasks[i].last = (int)((long long)units * (i + 1) / nthreads);
    pthread_create(&tid[i], NULL, recur_worker, &tasks[i]);
  }
  for (int i = 0; i < nthreads; ++i) pthread_join(tid[i], NULL);
  free(tid);
  free(tasks);
  return J.status;
}

/* ------------------------------------------------------------------------ */
/* Short causal convolution in front of the layer.                           */
/* ------------------------------------------------------------------------ */

/*
 * oracle_causal_conv -- depthwise causal convolution of width 4 per channel:
 *   y_t[c] = sum_{j=0..3} w[c, j] * x_{t-3+j}[c],
 * where x_{t'} for t' < 0 comes from cache_in (slot 3 + t'), or is zero when
 * cache_in is NULL.  cache_out (nullable) receives the last 3 inputs of the
 * concatenated history (cache, then x), oldest first, so that a following call
 * continues exactly where this one stopped; it may alias cache_in.
 */
int oracle_causal_conv(int B, int T, int Cch, const double *x, const double *w,
                       const double *cache_in, double *y, double *cache_out) {
  if (B < 0 || T < 0 || Cch <= 0) return ORACLE_EBADARG;
  double *hist = (double *)malloc(sizeof(double) * (size_t)(T + 3) * (Cch > 0 ? Cch : 1));
  if (!hist) return ORACLE_ENOMEM;
  for (int b = 0; b < B; ++b) {
    /* hist[s] = x_{s-3}: the 3 cached inputs followed by the T new ones */
    for (int s = 0; s < 3; ++s)
      for (int c = 0; c < Cch; ++c)
        hist[(size_t)s * Cch + c] = cache_in ? cache_in[((size_t)b * 3 + s) * Cch + c] : 0.0;
    for (int t = 0; t < T; ++t)
      for (int c = 0; c < Cch; ++c)
        hist[(size_t)(t + 3) * Cch + c] = x[((size_t)b * T + t) * Cch + c];
    for (int t = 0; t < T; ++t)
      for (int c = 0; c < Cch; ++c) {
        double acc = 0.0;
        for (int j = 0; j < 4; ++j) acc += w[(size_t)c * 4 + j] * hist[(size_t)(t + j) * Cch + c];
        y[((size_t)b * T + t) * Cch + c] = acc;
      }
    if (cache_out)
      for (int s = 0; s < 3; ++s)
        for (int c = 0; c < Cch; ++c)
          cache_out[((size_t)b * 3 + s) * Cch + c] = hist[(size_t)(T + s) * Cch + c];
  }
  free(hist);
  return ORACLE_OK;
}

/*
 * oracle_l2norm_rows -- x_r <- x_r / sqrt(sum x_r^2 + eps) for each of n rows
 * of length d, in place.  The Gated DeltaNet front end normalises q and k per
 * head so that the erase direction k_t has unit length.
 */
int oracle_l2norm_rows(long long n, int d, double *x, double eps) {
  if (n < 0 || d <= 0) return ORACLE_EBADARG;
  for (long long r = 0; r < n; ++r) {
    double *xr = x + r * d;
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += xr[i] * xr[i];
    const double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < d; ++i) xr[i] *= inv;
  }
  return ORACLE_OK;
}

/*
 * Single-precision front end.  With bf16 activations the convolution and the
 * L2 norm end in a rounding to bf16: the value decides an integer (the bf16
 * code), so this step is evaluated in the precision the layer computes its
 * front end in, single precision, in the order the definitions read:
 *   y = w0 x_{t-3} rounded, then each later tap added by one fused
 *       multiply-add (w1 x_{t-2}, w2 x_{t-1}, w3 x_t in turn: the exact
 *       product and sum, rounded once);
 *   s = sum of y_i^2 by pairwise summation (the row split in halves,
 *       recursively), every square and sum rounded on its own,
 *       r = 1 / sqrt(s + eps), y_i <- y_i r.
 * Inputs and outputs are doubles holding single-precision values.
 */
int oracle_causal_conv_f32(int B, int T, int Cch, const double *x, const double *w,
                           const double *cache_in, double *y, double *cache_out) {
  if (B < 0 || T < 0 || Cch <= 0) return ORACLE_EBADARG;
  float *hist = (float *)malloc(sizeof(float) * (size_t)(T + 3) * (size_t)Cch);
  if (!hist) return ORACLE_ENOMEM;
  for (int b = 0; b < B; ++b) {
    for (int s = 0; s < 3; ++s)
      for (int c = 0; c < Cch; ++c)
        hist[(size_t)s * Cch + c] = cache_in ? (float)cache_in[((size_t)b * 3 + s) * Cch + c] : 0.0f;
    for (int t = 0; t < T; ++t)
      for (int c = 0; c < Cch; ++c) hist[(size_t)(t + 3) * Cch + c] = (float)x[((size_t)b * T + t) * Cch + c];
    for (int t = 0; t < T; ++t)
      for (int c = 0; c < Cch; ++c) {
        float acc = (float)w[(size_t)c * 4] * hist[(size_t)t * Cch + c];
        for (int j = 1; j < 4; ++j) acc = fmaf((float)w[(size_t)c * 4 + j], hist[(size_t)(t + j) * Cch + c], acc);
        y[((size_t)b * T + t) * Cch + c] = (double)acc;
      }
    if (cache_out)
      for (int s = 0; s < 3; ++s)
        for (int c = 0; c < Cch; ++c)
          cache_out[((size_t)b * 3 + s) * Cch + c] = (double)hist[(size_t)(T + s) * Cch + c];
  }
  free(hist);
  return ORACLE_OK;
}

static float pairwise_sum_f32(const float *a, int n) {
  if (n == 1) return a[0];
  const int h = n / 2;
  return pairwise_sum_f32(a, h) + pairwise_sum_f32(a + h, n - h);
}

int oracle_l2norm_rows_f32(long long n, int d, double *x, double eps) {
  if (n < 0 || d <= 0) return ORACLE_EBADARG;
  float *sq = (float *)malloc(sizeof(float) * (size_t)d);
  if (!sq) return ORACLE_ENOMEM;
  const float epsf = (float)eps;
  for (long long r = 0; r < n; ++r) {
    double *xr = x + r * d;
    for (int i = 0; i < d; ++i) {
      const float v = (float)xr[i];
      sq[i] = v * v;
    }
    const float inv = 1.0f / sqrtf(pairwise_sum_f32(sq, d) + epsf);
    for (int i = 0; i < d; ++i) xr[i] = (double)((float)xr[i] * inv);
  }
  free(sq);
  return ORACLE_OK;
}

/*
 * oracle_round_bf16 -- round each value to the nearest bfloat16 (8 significant
 * bits, ties to even), in place, straight from double.  Activations enter the
 * layer in bf16 at deployment precision; finite normal range only.
 */
int oracle_round_bf16(long long n, double *x) {
  for (long long i = 0; i < n; ++i) {
    const double v = x[i];
    if (v == 0.0 || !isfinite(v)) continue;
    int e;
    const double m = frexp(v, &e);           /* v = m * 2^e, 0.5 <= |m| < 1 */
    const double r = nearbyint(ldexp(m, 8)); /* 8 significant bits, ties to even */
    x[i] = ldexp(r, e - 8);
  }
  return ORACLE_OK;
}
