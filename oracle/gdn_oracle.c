/*
 * gdn_oracle.c -- float64 CPU oracle of the Gated DeltaNet layer.
 *
 * TEST INFRASTRUCTURE ONLY (see gdn_oracle.h): plain loops in the order the
 * method defines them, token by token, no blocking, no chunking, no fusion.
 * Every floating-point step is done in double precision; inputs arrive as
 * float32 values (bf16 inputs are widened exactly before they get here).
 */
#include "gdn_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^{-z}).  (PicoLM changelog, "GPU:
 * Device-Native Pipeline Rewrite" lists the SiLU elementwise op; the conv
 * output of the linear-attention block goes through it.) */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* sigmoid(z) = 1 / (1 + e^{-z}) gives beta. */
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* softplus(z) = log(1 + e^z), written in the overflow-free form
 * max(z, 0) + log1p(e^{-|z|}), which is the same number. */
static double softplus(double z) {
  return (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z)));
}

/* Causal conv of one channel over one sequence, then SiLU.
 *   y_t = SiLU( sum_{w=0}^{W-1} wt[w] * xin(t - (W-1) + w) )
 * where xin(tau) = x[tau][c] for tau >= 0, the initial window row
 * (W-1)+tau for tau < 0 (oldest row first), or 0 without a window. */
static void conv_silu_channel(int64_t T, int64_t conv_dim, int64_t conv_w,
                              const float* x, const float* window0,
                              const float* conv_weight, int64_t c,
                              double* y, int64_t y_stride) {
  for (int64_t t = 0; t < T; ++t) {
    double acc = 0.0;
    for (int64_t w = 0; w < conv_w; ++w) {
      int64_t tau = t - (conv_w - 1) + w;
      double xv;
      if (tau >= 0) {
        xv = (double)x[tau * conv_dim + c];
      } else if (window0 != NULL) {
        xv = (double)window0[((conv_w - 1) + tau) * conv_dim + c];
      } else {
        xv = 0.0;
      }
      acc += (double)conv_weight[c * conv_w + w] * xv;
    }
    y[t * y_stride] = silu(acc);
  }
}

int oracle_conv_silu(int64_t T, int64_t conv_dim, int64_t conv_w,
                     const float* x, const float* window0,
                     const float* conv_weight, double* y) {
  if (T < 0 || conv_dim <= 0 || conv_w <= 0) return -1;
  for (int64_t c = 0; c < conv_dim; ++c)
    conv_silu_channel(T, conv_dim, conv_w, x, window0, conv_weight, c, y + c,
                      conv_dim);
  return 0;
}

int oracle_gdn_recurrence(int64_t T, int64_t d_k, int64_t d_v,
                          const double* qhat, const double* khat,
                          const double* v, const double* g,
                          const double* beta, const double* S0,
                          double* o, double* S_out) {
  if (T < 0 || d_k <= 0 || d_v <= 0) return -1;
  /* S is the math-convention memory, d_v rows by d_k columns: o = S q. */
  double* S = (double*)malloc(sizeof(double) * (size_t)(d_v * d_k));
  double* Sk = (double*)malloc(sizeof(double) * (size_t)d_v);
  if (!S || !Sk) {
    free(S);
    free(Sk);
    return -2;
  }
  for (int64_t e = 0; e < d_v * d_k; ++e) S[e] = S0 ? S0[e] : 0.0;

  for (int64_t t = 0; t < T; ++t) {
    const double* k = khat + t * d_k;
    const double* q = qhat + t * d_k;
    const double* vt = v + t * d_v;
    const double decay = exp(g[t]);
    const double bt = beta[t];
    /* S_{t-1} k */
    for (int64_t j = 0; j < d_v; ++j) {
      double acc = 0.0;
      for (int64_t i = 0; i < d_k; ++i) acc += S[j * d_k + i] * k[i];
      Sk[j] = acc;
    }
    /* S_t = e^{g} S_{t-1} (I - beta k k^T) + beta v k^T
     *     = e^{g} (S_{t-1} - beta (S_{t-1} k) k^T) + beta v k^T */
    for (int64_t j = 0; j < d_v; ++j) {
      for (int64_t i = 0; i < d_k; ++i) {
        double s = S[j * d_k + i];
        S[j * d_k + i] = decay * (s - bt * Sk[j] * k[i]) + bt * vt[j] * k[i];
      }
    }
    /* o_t = S_t q */
    for (int64_t j = 0; j < d_v; ++j) {
      double acc = 0.0;
      for (int64_t i = 0; i < d_k; ++i) acc += S[j * d_k + i] * q[i];
      o[t * d_v + j] = acc;
    }
  }
  for (int64_t e = 0; e < d_v * d_k; ++e) S_out[e] = S[e];
  free(S);
  free(Sk);
  return 0;
}

/* Scale every row of a [T][n] block to unit L2 norm (eps inside the root),
 * then multiply by `extra`. */
static void l2_normalise_rows(int64_t T, int64_t n, double eps, double extra,
                              double* rows) {
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += rows[t * n + i] * rows[t * n + i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int64_t i = 0; i < n; ++i) rows[t * n + i] *= inv * extra;
  }
}

int oracle_gdn_frontend_head(int64_t T, int64_t h_k, int64_t h_v,
                             int64_t d_k, int64_t d_v, int64_t conv_w,
                             int64_t h, const float* x, const float* a,
                             const float* b, const float* conv_weight,
                             const float* A_log, const float* dt_bias,
                             const float* window0, double l2_eps,
                             double* qhat, double* khat, double* v,
                             double* g, double* beta) {
  if (T < 0 || h_k <= 0 || h_v <= 0 || h_v % h_k != 0 || d_k <= 0 ||
      d_v <= 0 || conv_w <= 0 || h < 0 || h >= h_v)
    return -1;
  const int64_t conv_dim = 2 * h_k * d_k + h_v * d_v;
  const int64_t hk = h / (h_v / h_k); /* repeat-interleave expansion */
  const int64_t q0 = hk * d_k;                  /* q block of key head hk */
  const int64_t k0 = h_k * d_k + hk * d_k;      /* k block */
  const int64_t v0 = 2 * h_k * d_k + h * d_v;   /* v block of value head h */

  for (int64_t i = 0; i < d_k; ++i) {
    conv_silu_channel(T, conv_dim, conv_w, x, window0, conv_weight, q0 + i,
                      qhat + i, d_k);
    conv_silu_channel(T, conv_dim, conv_w, x, window0, conv_weight, k0 + i,
                      khat + i, d_k);
  }
  for (int64_t j = 0; j < d_v; ++j)
    conv_silu_channel(T, conv_dim, conv_w, x, window0, conv_weight, v0 + j,
                      v + j, d_v);

  l2_normalise_rows(T, d_k, l2_eps, 1.0 / sqrt((double)d_k), qhat);
  l2_normalise_rows(T, d_k, l2_eps, 1.0, khat);

  const double A = exp((double)A_log[h]);
  for (int64_t t = 0; t < T; ++t) {
    double z = (double)a[t * h_v + h] + (double)dt_bias[h];
    g[t] = -A * softplus(z);
    beta[t] = sigmoid((double)b[t * h_v + h]);
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Whole layer: one task per selected (sequence, value head).          */

typedef struct {
  int64_t h_k, h_v, d_k, d_v, conv_w, conv_dim;
  const float *x, *a, *b, *conv_weight, *A_log, *dt_bias, *window0, *state0;
  const int64_t* cu_seqlens;
  double l2_eps;
  double *o, *state_out;
  const int64_t* tasks; /* pairs (seq, head) */
  int64_t n_tasks;
  int64_t next;         /* next task index, guarded by mu */
  pthread_mutex_t mu;
  int err;
} layer_job;

static int run_task(layer_job* J, int64_t seq, int64_t h) {
  const int64_t start = J->cu_seqlens[seq];
  const int64_t T = J->cu_seqlens[seq + 1] - start;
  const int64_t d_k = J->d_k, d_v = J->d_v, h_v = J->h_v;
  double* qh = (double*)malloc(sizeof(double) * (size_t)((T ? T : 1) * d_k));
  double* kh = (double*)malloc(sizeof(double) * (size_t)((T ? T : 1) * d_k));
  double* vv = (double*)malloc(sizeof(double) * (size_t)((T ? T : 1) * d_v));
  double* gg = (double*)malloc(sizeof(double) * (size_t)(T ? T : 1));
  double* bb = (double*)malloc(sizeof(double) * (size_t)(T ? T : 1));
  double* oo = (double*)malloc(sizeof(double) * (size_t)((T ? T : 1) * d_v));
  double* S0 = (double*)malloc(sizeof(double) * (size_t)(d_v * d_k));
  double* S1 = (double*)malloc(sizeof(double) * (size_t)(d_v * d_k));
  int rc = 0;
  if (!qh || !kh || !vv || !gg || !bb || !oo || !S0 || !S1) {
    rc = -2;
    goto done;
  }
  const float* win = J->window0
                         ? J->window0 + seq * (J->conv_w - 1) * J->conv_dim
                         : NULL;
  rc = oracle_gdn_frontend_head(T, J->h_k, h_v, d_k, d_v, J->conv_w, h,
                                J->x + start * J->conv_dim,
                                J->a + start * h_v, J->b + start * h_v,
                                J->conv_weight, J->A_log, J->dt_bias, win,
                                J->l2_eps, qh, kh, vv, gg, bb);
  if (rc) goto done;
  /* stored initial state is S^T [d_k][d_v]; the recurrence wants S [d_v][d_k] */
  for (int64_t i = 0; i < d_k; ++i)
    for (int64_t j = 0; j < d_v; ++j)
      S0[j * d_k + i] =
          J->state0 ? (double)J->state0[((seq * h_v + h) * d_k + i) * d_v + j]
                    : 0.0;
  rc = oracle_gdn_recurrence(T, d_k, d_v, qh, kh, vv, gg, bb, S0, oo, S1);
  if (rc) goto done;
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < d_v; ++j)
      J->o[((start + t) * h_v + h) * d_v + j] = oo[t * d_v + j];
  for (int64_t i = 0; i < d_k; ++i)
    for (int64_t j = 0; j < d_v; ++j)
      J->state_out[((seq * h_v + h) * d_k + i) * d_v + j] = S1[j * d_k + i];
done:
  free(qh);
  free(kh);
  free(vv);
  free(gg);
  free(bb);
  free(oo);
  free(S0);
  free(S1);
  return rc;
}

static void* worker(void* arg) {
  layer_job* J = (layer_job*)arg;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t idx = J->next++;
    int stop = idx >= J->n_tasks || J->err;
    pthread_mutex_unlock(&J->mu);
    if (stop) break;
    int rc = run_task(J, J->tasks[2 * idx], J->tasks[2 * idx + 1]);
    if (rc) {
      pthread_mutex_lock(&J->mu);
      J->err = rc;
      pthread_mutex_unlock(&J->mu);
    }
  }
  return NULL;
}

int oracle_gdn_layer(int64_t h_k, int64_t h_v, int64_t d_k, int64_t d_v,
                     int64_t conv_w, const float* x, const float* a,
                     const float* b, const float* conv_weight,
                     const float* A_log, const float* dt_bias,
                     const int64_t* cu_seqlens, int64_t num_seqs,
                     const float* window0, const float* state0,
                     const uint8_t* head_mask, double l2_eps,
                     double* o, double* state_out, double* window_out,
                     int n_threads) {
  if (h_k <= 0 || h_v <= 0 || h_v % h_k != 0 || d_k <= 0 || d_v <= 0 ||
      conv_w <= 0 || num_seqs < 0 || !cu_seqlens || !o || !state_out)
    return -1;
  if (cu_seqlens[0] != 0) return -1;
  for (int64_t s = 0; s < num_seqs; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
  const int64_t conv_dim = 2 * h_k * d_k + h_v * d_v;

  /* Final conv window of every sequence: the last W-1 raw inputs, oldest
   * first; rows before the sequence start come from the initial window. */
  if (window_out) {
    for (int64_t s = 0; s < num_seqs; ++s) {
      const int64_t start = cu_seqlens[s];
      const int64_t T = cu_seqlens[s + 1] - start;
      for (int64_t r = 0; r < conv_w - 1; ++r) {
        int64_t tau = T - (conv_w - 1) + r; /* position within the sequence */
        for (int64_t c = 0; c < conv_dim; ++c) {
          double xv;
          if (tau >= 0)
            xv = (double)x[(start + tau) * conv_dim + c];
          else if (window0)
            xv = (double)window0[(s * (conv_w - 1) + (conv_w - 1) + tau) *
                                     conv_dim + c];
          else
            xv = 0.0;
          window_out[(s * (conv_w - 1) + r) * conv_dim + c] = xv;
        }
      }
    }
  }

  int64_t n_tasks = 0;
  for (int64_t s = 0; s < num_seqs; ++s)
    for (int64_t h = 0; h < h_v; ++h)
      if (!head_mask || head_mask[s * h_v + h]) ++n_tasks;
  int64_t* tasks = (int64_t*)malloc(sizeof(int64_t) * (size_t)(2 * (n_tasks + 1)));
  if (!tasks) return -2;
  int64_t k = 0;
  for (int64_t s = 0; s < num_seqs; ++s)
    for (int64_t h = 0; h < h_v; ++h)
      if (!head_mask || head_mask[s * h_v + h]) {
        tasks[2 * k] = s;
        tasks[2 * k + 1] = h;
        ++k;
      }

  layer_job J;
  memset(&J, 0, sizeof(J));
  J.h_k = h_k; J.h_v = h_v; J.d_k = d_k; J.d_v = d_v;
  J.conv_w = conv_w; J.conv_dim = conv_dim;
  J.x = x; J.a = a; J.b = b; J.conv_weight = conv_weight;
  J.A_log = A_log; J.dt_bias = dt_bias;
  J.window0 = window0; J.state0 = state0;
  J.cu_seqlens = cu_seqlens; J.l2_eps = l2_eps;
  J.o = o; J.state_out = state_out;
  J.tasks = tasks; J.n_tasks = n_tasks; J.next = 0; J.err = 0;
  pthread_mutex_init(&J.mu, NULL);

  if (n_threads < 1) n_threads = 1;
  if (n_threads > 1024) n_threads = 1024;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  int started = 0;
  if (th) {
    for (int i = 0; i < n_threads; ++i) {
      if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
      ++started;
    }
  }
  if (started == 0) worker(&J); /* no thread could start: run inline */
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&J.mu);
  free(tasks);
  return J.err;
}

/* ------------------------------------------------------------------ */
/* Gated RMSNorm of the layer output (the DeltaNet "gated norm").     */
/* Per row of d_v values (one token, one value head):                 */
/*   y_j = o_j / sqrt(mean_j o_j^2 + eps) * w_j * SiLU(z_j)            */
/* The weight is applied as stored: of the model's norms only this    */
/* one carries no pre-added +1 (oxydllm 0.0.0-alpha.12.2 release      */
/* notes, New Features, "GGUF qwen35 architecture"); the gated RMSNorm */
/* runs over the whole token batch after the scan ("Gated DeltaNet    */
/* fast paths").  The mean runs over the head's d_v values.           */
int oracle_gated_rmsnorm(int64_t rows, int64_t d_v, const float* o, const float* z,
                         const float* w, double eps, double* y) {
  if (rows < 0 || d_v <= 0 || !o || !z || !w || !y) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    const float* orow = o + r * d_v;
    const float* zrow = z + r * d_v;
    double ss = 0.0;
    for (int64_t j = 0; j < d_v; ++j) ss += (double)orow[j] * (double)orow[j];
    const double inv = 1.0 / sqrt(ss / (double)d_v + eps);
    for (int64_t j = 0; j < d_v; ++j)
      y[r * d_v + j] = (double)orow[j] * inv * (double)w[j] * silu((double)zrow[j]);
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* The decay and beta input projections as one matmul (oxydllm notes, */
/* Performance, "Gated DeltaNet fast paths": the small beta/decay     */
/* projections fuse into one matmul).  With W = [W_a; W_b], 2 h_v     */
/* rows of d_model weights:                                           */
/*   a[t][h] = sum_i hidden[t][i] W[h][i]         (decay input)       */
/*   b[t][h] = sum_i hidden[t][i] W[h_v + h][i]   (beta input)        */
/* for every token t and value head h < h_v, summed in index order.   */
int oracle_gate_projection(int64_t n, int64_t d_model, int64_t h_v, const float* hidden,
                           const float* w, double* a, double* b) {
  if (n < 0 || d_model <= 0 || h_v <= 0 || !hidden || !w || !a || !b) return -1;
  for (int64_t t = 0; t < n; ++t) {
    const float* x = hidden + t * d_model;
    for (int64_t r = 0; r < 2 * h_v; ++r) {
      const float* wr = w + r * d_model;
      double acc = 0.0;
      for (int64_t i = 0; i < d_model; ++i) acc += (double)x[i] * (double)wr[i];
      if (r < h_v) a[t * h_v + r] = acc;
      else b[t * h_v + (r - h_v)] = acc;
    }
  }
  return 0;
}
