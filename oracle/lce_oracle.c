/*
 * Plain-C fp64 oracle for the fused LM-head linear + cross-entropy.
 * TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library; the product path never does.
 *
 * It is an independent second implementation of the definition that
 * lce_oracle.py writes out with numpy (the token-level cross-entropy of the
 * LM-head logits and its gradients, "XTuner on Ascend 910C: Qwen3.5-2B
 * training optimisation", section 3.1.4): plain loops, no BLAS, no blocking.
 *
 *   pass A (rows in parallel):  z_i = H_i W^T, lse_i, loss_i, G_i, dH_i = G_i W
 *   pass B (vocab rows in parallel): z_{.v} recomputed, dW_v = sum_i G_iv H_i
 *
 * Each output element is written by exactly one thread and every sum runs in
 * a fixed index order, so results are deterministic for any thread count.
 * Inputs are bf16 bit patterns widened exactly to fp64.
 *
 * Return codes: 0 ok, 1 invalid argument, 2 label outside {ignore} U [0, V),
 * 3 out of host memory.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const double *H, *W;     /* decoded inputs [N,d], [V,d] */
  const int64_t *y;
  int64_t N, d, V, ignore_index;
  double gscale;           /* g/n (mean) or g (sum); 0 when n = 0 under mean */
  double *lse, *loss_i, *dH, *dW;
  int64_t lo, hi;          /* this worker's share of rows (pass A) or vocab rows (pass B) */
} job_t;

static void *pass_rows(void *arg) {
  job_t *j = (job_t *)arg;
  double *z = (double *)malloc(sizeof(double) * (size_t)j->V);
  if (!z) return (void *)1;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    const double *h = j->H + i * j->d;
    double m = -INFINITY;
    for (int64_t v = 0; v < j->V; ++v) {
      const double *w = j->W + v * j->d;
      double acc = 0.0;
      for (int64_t k = 0; k < j->d; ++k) acc += h[k] * w[k];
      z[v] = acc;
      if (acc > m) m = acc;
    }
    double s = 0.0;
    for (int64_t v = 0; v < j->V; ++v) s += exp(z[v] - m);
    double lse = m + log(s);
    j->lse[i] = lse;
    int valid = j->y[i] != j->ignore_index;
    j->loss_i[i] = valid ? lse - z[j->y[i]] : 0.0;
    double *dh = j->dH + i * j->d;
    for (int64_t k = 0; k < j->d; ++k) dh[k] = 0.0;
    if (!valid) continue;
    for (int64_t v = 0; v < j->V; ++v) {
      double g = exp(z[v] - lse) - (v == j->y[i] ? 1.0 : 0.0);
      g *= j->gscale;
      const double *w = j->W + v * j->d;
      for (int64_t k = 0; k < j->d; ++k) dh[k] += g * w[k];
    }
  }
  free(z);
  return NULL;
}

static void *pass_vocab(void *arg) {
  job_t *j = (job_t *)arg;
  for (int64_t v = j->lo; v < j->hi; ++v) {
    const double *w = j->W + v * j->d;
    double *dw = j->dW + v * j->d;
    for (int64_t k = 0; k < j->d; ++k) dw[k] = 0.0;
    for (int64_t i = 0; i < j->N; ++i) {
      if (j->y[i] == j->ignore_index) continue;
      const double *h = j->H + i * j->d;
      double z = 0.0;
      for (int64_t k = 0; k < j->d; ++k) z += h[k] * w[k];
      double g = exp(z - j->lse[i]) - (v == j->y[i] ? 1.0 : 0.0);
      g *= j->gscale;
      for (int64_t k = 0; k < j->d; ++k) dw[k] += g * h[k];
    }
  }
  return NULL;
}

static int run_pass(void *(*fn)(void *), job_t *proto, int64_t total, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  job_t jobs[256];
  int rc = 0;
  int64_t per = (total + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *proto;
    jobs[t].lo = t * per < total ? t * per : total;
    jobs[t].hi = (t + 1) * per < total ? (t + 1) * per : total;
    if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0) { rc = 3; break; }
    ++started;
  }
  for (int t = 0; t < started; ++t) {
    void *r = NULL;
    pthread_join(th[t], &r);
    if (r) rc = 3;
  }
  return rc;
}

/*
 * reduction: 0 = mean over valid tokens, 1 = sum.
 * n_valid_override < 0: count valid labels; otherwise use it as the denominator.
 * grad_loss: upstream gradient g of the scalar loss.
 * Outputs (all fp64, caller-allocated): loss[1], lse[N], loss_i[N], dH[N*d],
 * dW[V*d]; dH/dW may be NULL to skip the backward (pass B is then skipped).
 */
int lce_oracle_f64(const uint16_t *Hbits, const uint16_t *Wbits, const int64_t *y,
                   int64_t N, int64_t d, int64_t V, int64_t ignore_index,
                   int reduction, int64_t n_valid_override, double grad_loss,
                   int nthreads, double *loss, double *lse, double *loss_i,
                   double *dH, double *dW) {
  if (!Hbits || !Wbits || !y || !loss || !lse || !loss_i) return 1;
  if (N < 0 || d <= 0 || V <= 0 || (reduction != 0 && reduction != 1)) return 1;
  for (int64_t i = 0; i < N; ++i)
    if (y[i] != ignore_index && (y[i] < 0 || y[i] >= V)) return 2;

  int64_t n = 0;
  for (int64_t i = 0; i < N; ++i) n += (y[i] != ignore_index);
  if (n_valid_override >= 0) n = n_valid_override;
  double lscale, gscale;
  if (reduction == 0) {
    lscale = n ? 1.0 / (double)n : 0.0;
    gscale = n ? grad_loss / (double)n : 0.0;
  } else {
    lscale = 1.0;
    gscale = grad_loss;
  }

  double *Hd = (double *)malloc(sizeof(double) * (size_t)(N * d + 1));
  double *Wd = (double *)malloc(sizeof(double) * (size_t)(V * d));
  double *dHtmp = dH ? NULL : (double *)malloc(sizeof(double) * (size_t)(N * d + 1));
  if (!Hd || !Wd || (!dH && !dHtmp)) { free(Hd); free(Wd); free(dHtmp); return 3; }
  for (int64_t e = 0; e < N * d; ++e) Hd[e] = bf16_to_f64(Hbits[e]);
  for (int64_t e = 0; e < V * d; ++e) Wd[e] = bf16_to_f64(Wbits[e]);

  job_t proto;
  memset(&proto, 0, sizeof proto);
  proto.H = Hd; proto.W = Wd; proto.y = y;
  proto.N = N; proto.d = d; proto.V = V; proto.ignore_index = ignore_index;
  proto.gscale = gscale; proto.lse = lse; proto.loss_i = loss_i;
  proto.dH = dH ? dH : dHtmp; proto.dW = dW;

  int rc = run_pass(pass_rows, &proto, N, nthreads);
  if (rc == 0 && dW) rc = run_pass(pass_vocab, &proto, V, nthreads);

  double acc = 0.0;
  for (int64_t i = 0; i < N; ++i) acc += loss_i[i];
  *loss = acc * lscale;

  free(Hd); free(Wd); free(dHtmp);
  return rc;
}
