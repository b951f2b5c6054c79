/*
 * gdn_oracle.h -- float64 CPU oracle of the Gated DeltaNet (gated delta rule)
 * linear-attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This code exists to check the CUDA library
 * against a plain, slow, obviously correct restatement of the method.  Only
 * the test suite, the smoke check of the package entry point and the CPU
 * baseline leg of the benchmark may load it.  The CUDA library never includes
 * this header or links this code, and this code shares nothing with it.
 *
 * What is computed (per sequence, per value head h, token by token):
 *
 *   causal conv:  y_t[c] = sum_{w=0}^{W-1} Wc[c][w] * x_{t-(W-1)+w}[c],
 *                 x_tau for tau < 0 taken from the initial window (oldest
 *                 row first) or zero;  then SiLU(y) = y * sigmoid(y).
 *                 (Vallmo README, "What's here": causal conv1d kernel;
 *                  oxydllm 0.0.0-alpha.12.2 release notes, New Features,
 *                  "Gated DeltaNet runtime": the causal-conv window that is
 *                  kept per sequence.)
 *   split:        y = q | k | v, each head-major; q,k have H_k heads of d_k,
 *                 v has H_v heads of d_v; value head h reads key head
 *                 h / (H_v / H_k) (repeat-interleave expansion; the oxydllm
 *                 notes, New Features, "GGUF qwen35 architecture", contrast
 *                 this with the tiled order a GGUF file stores).
 *   normalise:    q^ = q / sqrt(sum q^2 + eps) / sqrt(d_k),
 *                 k^ = k / sqrt(sum k^2 + eps)
 *                 (PicoLM changelog, "GPU: Device-Native Pipeline Rewrite":
 *                  the l2norm step of the SSM kernels).
 *   gates:        g_t = -exp(A_log[h]) * softplus(a_t[h] + dt_bias[h]),
 *                 beta_t = sigmoid(b_t[h])
 *                 (oxydllm notes, New Features: ssm_a is the negated
 *                  exponential of A_log; the scalar parameters stay F32).
 *   recurrence:   S_t = exp(g_t) * S_{t-1} (I - beta_t k^_t k^_t^T)
 *                       + beta_t v_t k^_t^T,      o_t = S_t q^_t
 *                 with S a d_v x d_k matrix (Gated DeltaNet, the published
 *                 gated delta rule the valkyr README names as prior art in
 *                 its License section; the 32x128x128 F32 memory of the
 *                 oxydllm notes, New Features, "Gated DeltaNet runtime").
 *
 * Layouts (all row-major, C order):
 *   x            [T_tot][conv_dim]  float32 (bf16 inputs arrive widened)
 *   a, b         [T_tot][H_v]       float32
 *   conv_weight  [conv_dim][W]      float32, tap W-1 multiplies the current token
 *   A_log, dt_bias [H_v]            float32
 *   window0      [num_seqs][W-1][conv_dim] float32, oldest row first, or NULL
 *   state0       [num_seqs][H_v][d_k][d_v] float32 (S transposed), or NULL
 *   o            [T_tot][H_v][d_v]  float64
 *   state_out    [num_seqs][H_v][d_k][d_v] float64 (S transposed)
 *   window_out   [num_seqs][W-1][conv_dim] float64
 * The math-convention state S[d_v][d_k] is used inside; storage is S^T so the
 * value index is contiguous.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Core recurrence for one head.  qhat, khat [T][d_k]; v [T][d_v]; g, beta [T].
 * S0 / S_out in math layout [d_v][d_k]; S0 may be NULL (zero state).
 * o [T][d_v].  Returns 0. */
int oracle_gdn_recurrence(int64_t T, int64_t d_k, int64_t d_v,
                          const double* qhat, const double* khat,
                          const double* v, const double* g,
                          const double* beta, const double* S0,
                          double* o, double* S_out);

/* Front end of one sequence for one value head h: conv + SiLU, split,
 * L2 normalisation with the 1/sqrt(d_k) query scale, gates.
 * x points at the sequence's first row (row stride conv_dim).
 * Outputs qhat, khat [T][d_k], v [T][d_v], g, beta [T].  Returns 0, or -1 on
 * bad dimensions. */
int oracle_gdn_frontend_head(int64_t T, int64_t h_k, int64_t h_v,
                             int64_t d_k, int64_t d_v, int64_t conv_w,
                             int64_t h, const float* x, const float* a,
                             const float* b, const float* conv_weight,
                             const float* A_log, const float* dt_bias,
                             const float* window0, double l2_eps,
                             double* qhat, double* khat, double* v,
                             double* g, double* beta);

/* Conv + SiLU for every channel of one sequence: y [T][conv_dim]. */
int oracle_conv_silu(int64_t T, int64_t conv_dim, int64_t conv_w,
                     const float* x, const float* window0,
                     const float* conv_weight, double* y);

/* Whole varlen layer.  cu_seqlens [num_seqs+1] (host).  head_mask
 * [num_seqs][H_v] selects the (sequence, head) pairs to compute (NULL = all);
 * outputs of unselected pairs are left untouched.  window_out may be NULL.
 * n_threads >= 1 worker threads split the selected pairs.
 * Returns 0, or -1 on bad arguments. */
int oracle_gdn_layer(int64_t h_k, int64_t h_v, int64_t d_k, int64_t d_v,
                     int64_t conv_w, const float* x, const float* a,
                     const float* b, const float* conv_weight,
                     const float* A_log, const float* dt_bias,
                     const int64_t* cu_seqlens, int64_t num_seqs,
                     const float* window0, const float* state0,
                     const uint8_t* head_mask, double l2_eps,
                     double* o, double* state_out, double* window_out,
                     int n_threads);

/* Gated RMSNorm over rows of d_v values: y [rows][d_v] float64 from o, z
 * [rows][d_v] and the per-channel weight w [d_v] (applied as stored).
 * Returns 0, or -1 on bad arguments. */
int oracle_gated_rmsnorm(int64_t rows, int64_t d_v, const float* o, const float* z,
                         const float* w, double eps, double* y);

/* The decay and beta input projections as one matmul: hidden [n][d_model]
 * and W [2 h_v][d_model] (rows 0 .. h_v - 1 the decay projection W_a, rows
 * h_v .. 2 h_v - 1 the beta projection W_b) give a = hidden W_a^T and
 * b = hidden W_b^T, each [n][h_v] float64.  Returns 0, or -1 on bad
 * arguments. */
int oracle_gate_projection(int64_t n, int64_t d_model, int64_t h_v, const float* hidden,
                           const float* w, double* a, double* b);

#ifdef __cplusplus
}
#endif

#endif /* GDN_ORACLE_H */
