// gdn_prefill_simt.cu -- chunked prefill of the Gated DeltaNet layer on the
// fp32 SIMT pipes, for every supported shape (d_k, d_v in {16,32,64,128},
// chunk in {16,32,64,128}, fp32 or bf16 I/O).  The tensor-core path takes the
// Qwen3.5-4B layer shape; this path serves the other shapes and fp32 I/O, whose
// 1e-3 tolerance bf16 tensor-core operands would not meet.
//
// Kernels, in stream order:
//   1. check_cu_seqlens   one CTA; sets the workspace flag (and the device
//                         status bit when cu_seqlens is malformed) and writes
//                         the chunk table (each sequence's first chunk).
//   2. frontend           one CTA per token: causal conv (window or zero
//                         history before the sequence start) + SiLU, L2 norm
//                         of q and k with the 1/sqrt(d_k) query scale, gates.
//   3. window_writeback   the last W-1 raw inputs of each sequence to its slot.
//   4. chunk              one CTA per (chunk, value head), all chunks at once:
//                         the state-independent factors of the chunked WY form
//                         (oxydllm 0.0.0-alpha.12.2 release notes, New
//                         Features, "Gated DeltaNet runtime": chunked parallel
//                         scan, per-chunk unit-lower-triangular system), with
//                         gamma the cumulative log-decay inside the chunk:
//       A = strict_tril(diag(beta) K K^T * e^{gamma_r - gamma_s})
//       T = (I + A)^-1           (column-wise forward substitution: exact
//                                 entries, no matrix powers, finite on fully
//                                 correlated keys)
//       U = T diag(beta) V,  Wk = T diag(beta e^gamma) K,
//       P = tril(Q K^T * e^{gamma_r - gamma_s})
//   5. scan               one CTA per (sequence, value head, d_v tile),
//                         sequential over chunks, state in shared memory
//                         (the chunk inputs streamed through two buffers where
//                         they would not fit side by side):
//       W = U - Wk S^T
//       O = diag(e^gamma) Q S^T + P W
//       S^T <- e^{gamma_last} S^T + K^T diag(e^{gamma_last - gamma}) W
//     Only e^{x} with x <= 0 is ever formed.  The products run as register
//     blocks of 2 x 4 to 8 x 4 per thread on shared-memory operands.
#include <type_traits>

#include "gdn_common.cuh"

namespace gdn {

// Also, when chunk_off is given and cu_seqlens is valid, the first global
// chunk of each sequence: chunk_off[b] = sum_{b' < b} ceil(len_b' / chunk),
// chunk_off[num_seqs] = the number of chunks.
__global__ void __launch_bounds__(256) check_cu_seqlens_kernel(const int32_t* __restrict__ cu,
                                                               int num_seqs, int64_t total,
                                                               int chunk, int32_t* chunk_off,
                                                               int32_t* flag, int32_t* d_status) {
  __shared__ int bad;
  __shared__ int part[256];
  if (threadIdx.x == 0) bad = (cu[0] != 0) || ((int64_t)cu[num_seqs] != total);
  __syncthreads();
  for (int i = threadIdx.x; i < num_seqs; i += blockDim.x)
    if (cu[i + 1] < cu[i]) bad = 1;
  __syncthreads();
  if (chunk_off && !bad) {   // bad is the same for every thread here
    const int per = (num_seqs + (int)blockDim.x - 1) / (int)blockDim.x;
    const int b0 = min(num_seqs, (int)threadIdx.x * per), b1 = min(num_seqs, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += (int)(((int64_t)cu[b + 1] - cu[b] + chunk - 1) / chunk);
    part[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
      int run = 0;
      for (int i = 0; i < (int)blockDim.x; ++i) {
        const int v = part[i];
        part[i] = run;
        run += v;
      }
      chunk_off[num_seqs] = run;
    }
    __syncthreads();
    int run = part[threadIdx.x];
    for (int b = b0; b < b1; ++b) {
      chunk_off[b] = run;
      run += (int)(((int64_t)cu[b + 1] - cu[b] + chunk - 1) / chunk);
    }
  }
  if (threadIdx.x == 0) {
    flag[0] = bad ? 0 : 1;
    if (bad) set_status(d_status, GDN_DEV_BAD_CU_SEQLENS);
  }
}

// Sequence of token t: the b with cu[b] <= t < cu[b+1] (zero-length
// sequences skipped).
__device__ __forceinline__ int seq_of_token(const int32_t* __restrict__ cu, int num_seqs, int64_t t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Eight consecutive values of the I/O type as floats (16-byte aligned source).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename IO>
__global__ void __launch_bounds__(256) frontend_kernel(const GdnPrefillArgs args) {
  extern __shared__ float s_y[];  // [conv_dim]
  if (!args.ws_flag[0]) return;
  const int64_t tok = blockIdx.x;
  const int b = seq_of_token(args.cu_seqlens, args.num_seqs, tok);
  const int slot = args.slot_idx[b];
  if (slot < 0 || slot >= args.num_slots) return;  // status set by the scan
  const int64_t p = tok - args.cu_seqlens[b];       // position in the sequence
  const bool init = args.has_init ? args.has_init[b] != 0 : false;
  const int cd = args.conv_dim;
  const IO* __restrict__ x = reinterpret_cast<const IO*>(args.x);
  const IO* __restrict__ win = reinterpret_cast<const IO*>(args.conv_pool) + (size_t)slot * 3 * cd;

  // eight channels per thread, 16-byte loads (conv_dim is a multiple of 16)
  for (int c = 8 * threadIdx.x; c < cd; c += 8 * blockDim.x) {
    float xv[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t tau = p - 3 + k;  // position of this tap's input
      if (tau >= 0) load8(x + (size_t)(tok - 3 + k) * cd + c, xv[k]);
      else if (init) load8(win + (size_t)(3 + tau) * cd + c, xv[k]);
      else
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[k][e] = 0.f;
    }
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 w = *reinterpret_cast<const float4*>(args.conv_weight + 4 * (size_t)(c + e));
      float z = w.x * xv[0][e];   // taps oldest first
      z = fmaf(w.y, xv[1][e], z);
      z = fmaf(w.z, xv[2][e], z);
      z = fmaf(w.w, xv[3][e], z);
      y[e] = silu(z);
    }
    *reinterpret_cast<float4*>(s_y + c) = make_float4(y[0], y[1], y[2], y[3]);
    *reinterpret_cast<float4*>(s_y + c + 4) = make_float4(y[4], y[5], y[6], y[7]);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  // q and k heads: 2*h_k rows of d_k channels, one warp per head
  for (int hh = warp; hh < 2 * args.h_k; hh += nw) {
    const float* y = s_y + (size_t)hh * args.d_k;
    float ss = 0.f;
    for (int i = lane; i < args.d_k; i += 32) ss = fmaf(y[i], y[i], ss);
    ss = warp_sum(ss);
    const bool is_q = hh < args.h_k;
    const float scale = rsqrtf(ss + args.l2_eps) * (is_q ? rsqrtf((float)args.d_k) : 1.0f);
    float* dst = (is_q ? args.ws_q + (size_t)(tok * args.h_k + hh) * args.d_k
                       : args.ws_k + (size_t)(tok * args.h_k + (hh - args.h_k)) * args.d_k);
    for (int i = lane; i < args.d_k; i += 32) dst[i] = y[i] * scale;
  }
  const int v0 = 2 * args.h_k * args.d_k;
  for (int e = threadIdx.x; e < args.h_v * args.d_v; e += blockDim.x)
    args.ws_v[(size_t)tok * args.h_v * args.d_v + e] = s_y[v0 + e];
  for (int h = threadIdx.x; h < args.h_v; h += blockDim.x) {
    const float av = ld_io(reinterpret_cast<const IO*>(args.a) + (size_t)tok * args.h_v + h);
    const float bv = ld_io(reinterpret_cast<const IO*>(args.b) + (size_t)tok * args.h_v + h);
    args.ws_g[(size_t)tok * args.h_v + h] = gate_g(av, args.A_log[h], args.dt_bias[h]);
    args.ws_beta[(size_t)tok * args.h_v + h] = sigmoidf_(bv);
  }
}

// New window of each sequence: rows r = 0..W-2 hold the input at position
// T - (W-1) + r, from x when >= 0, else from the old window (row T + r) or 0.
template <typename IO>
__global__ void __launch_bounds__(256) window_writeback_kernel(const GdnPrefillArgs args) {
  if (!args.ws_flag[0]) return;
  const int b = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= args.conv_dim) return;
  const int slot = args.slot_idx[b];
  if (slot < 0 || slot >= args.num_slots) return;
  const int64_t start = args.cu_seqlens[b];
  const int64_t T = args.cu_seqlens[b + 1] - start;
  const bool init = args.has_init ? args.has_init[b] != 0 : false;
  const int cd = args.conv_dim;
  const IO* __restrict__ x = reinterpret_cast<const IO*>(args.x);
  if (blockIdx.z > 0) {
    // windows of the interval checkpoints k = z, z + (gridDim.z - 1), ...: the
    // three raw inputs before position k * every (every >= 16 tokens > 3, so all
    // inside the sequence)
    const int64_t every = (int64_t)args.ckpt_every_chunks * args.chunk;
    for (int64_t k = blockIdx.z; k * every < T; k += gridDim.z - 1) {
      const int64_t cs = ckpt_slot_of(args, b, k * args.ckpt_every_chunks, T);
      if (cs < 0) continue;
      IO* cw = reinterpret_cast<IO*>(args.conv_pool) + (size_t)cs * 3 * cd;
      IO v[3];
#pragma unroll
      for (int r = 0; r < 3; ++r) v[r] = x[(size_t)(start + k * every - 3 + r) * cd + c];
#pragma unroll
      for (int r = 0; r < 3; ++r) cw[(size_t)r * cd + c] = v[r];
    }
    return;
  }
  IO* win = reinterpret_cast<IO*>(args.conv_pool) + (size_t)slot * 3 * cd;
  IO vals[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int64_t tau = T - 3 + r;
    if (tau >= 0) vals[r] = x[(size_t)(start + tau) * cd + c];
    else if (init) vals[r] = win[(size_t)(T + r) * cd + c];
    else st_io(&vals[r], 0.0f);
  }
#pragma unroll
  for (int r = 0; r < 3; ++r) win[(size_t)r * cd + c] = vals[r];
}

// ---- register-tiled products on shared-memory operands -----------------------
// Each thread accumulates an RM x RN block: acc[m][n] += sum_k a(m, k) b(k, n).
// "rows" operands are read one float per row (rows padded to d + 4 floats, so
// consecutive rows start four banks apart); "cols" operands four floats at a
// time from 16-byte aligned rows; sc, when given, scales b's row k.

// a(m, k) = A[(r0 + m st) * lda + k], b(k, n) = B[(c0 + n st) * ldb + k] (both
// by rows, rows st apart: the lanes of a warp then read consecutive rows)
template <int RM, int RN>
__device__ __forceinline__ void tile_rows_rows(float (&acc)[RM][RN], const float* A, int lda,
                                               int r0, const float* B, int ldb, int c0, int st,
                                               int K) {
  for (int k = 0; k < K; ++k) {
    float a[RM], b[RN];
#pragma unroll
    for (int m = 0; m < RM; ++m) a[m] = A[(r0 + m * st) * lda + k];
#pragma unroll
    for (int n = 0; n < RN; ++n) b[n] = B[(c0 + n * st) * ldb + k];
#pragma unroll
    for (int m = 0; m < RM; ++m)
#pragma unroll
      for (int n = 0; n < RN; ++n) acc[m][n] = fmaf(a[m], b[n], acc[m][n]);
  }
}

// a(m, k) = A[(r0 + m) * lda + k] (by rows), b(k, n) = sc[k] B[k * ldb + c0 + n] (by columns)
template <int RM, int RN>
__device__ __forceinline__ void tile_rows_cols(float (&acc)[RM][RN], const float* A, int lda,
                                               int r0, const float* B, int ldb, int c0, int k0,
                                               int k1, const float* sc) {
  static_assert(RN % 4 == 0, "four columns per load");
  for (int k = k0; k < k1; ++k) {
    float a[RM], b[RN];
#pragma unroll
    for (int m = 0; m < RM; ++m) a[m] = A[(r0 + m) * lda + k];
    const float s = sc ? sc[k] : 1.0f;
#pragma unroll
    for (int n = 0; n < RN; n += 4) {
      const float4 v = *reinterpret_cast<const float4*>(B + k * ldb + c0 + n);
      b[n] = v.x * s; b[n + 1] = v.y * s; b[n + 2] = v.z * s; b[n + 3] = v.w * s;
    }
#pragma unroll
    for (int m = 0; m < RM; ++m)
#pragma unroll
      for (int n = 0; n < RN; ++n) acc[m][n] = fmaf(a[m], b[n], acc[m][n]);
  }
}

// a(m, k) = A[k * lda + r0 + m], b(k, n) = sc[k] B[k * ldb + c0 + n] (both by columns)
template <int RM, int RN>
__device__ __forceinline__ void tile_cols_cols(float (&acc)[RM][RN], const float* A, int lda,
                                               int r0, const float* B, int ldb, int c0, int K,
                                               const float* sc) {
  static_assert(RM % 4 == 0 && RN % 4 == 0, "four rows and columns per load");
  for (int k = 0; k < K; ++k) {
    float a[RM], b[RN];
#pragma unroll
    for (int m = 0; m < RM; m += 4) {
      const float4 v = *reinterpret_cast<const float4*>(A + k * lda + r0 + m);
      a[m] = v.x; a[m + 1] = v.y; a[m + 2] = v.z; a[m + 3] = v.w;
    }
    const float s = sc[k];
#pragma unroll
    for (int n = 0; n < RN; n += 4) {
      const float4 v = *reinterpret_cast<const float4*>(B + k * ldb + c0 + n);
      b[n] = v.x * s; b[n + 1] = v.y * s; b[n + 2] = v.z * s; b[n + 3] = v.w * s;
    }
#pragma unroll
    for (int m = 0; m < RM; ++m)
#pragma unroll
      for (int n = 0; n < RN; ++n) acc[m][n] = fmaf(a[m], b[n], acc[m][n]);
  }
}

// a(m, k) = T[r0 + m][k] for the unit lower-triangular T stored transposed in
// the upper triangle (and diagonal) of AT: T[r][k] = AT[k * lda + r] for k <= r,
// 0 for k > r (AT holds A there); b(k, n) = sc[k] B[k * ldb + c0 + n].  Four
// rows r0 .. r0 + 3 (r0 a multiple of 4), k over 0 .. r0 + 3.
template <int RN>
__device__ __forceinline__ void tile_tt_cols(float (&acc)[4][RN], const float* AT, int lda, int r0,
                                             const float* B, int ldb, int c0, const float* sc) {
  static_assert(RN % 4 == 0, "four columns per load");
  for (int k = 0; k < r0 + 4; ++k) {
    const float4 v = *reinterpret_cast<const float4*>(AT + k * lda + r0);
    float a[4] = {v.x, v.y, v.z, v.w};
    if (k > r0) {
#pragma unroll
      for (int m = 0; m < 4; ++m) a[m] = m < k - r0 ? 0.f : a[m];
    }
    const float s = sc[k];
    float b[RN];
#pragma unroll
    for (int n = 0; n < RN; n += 4) {
      const float4 w = *reinterpret_cast<const float4*>(B + k * ldb + c0 + n);
      b[n] = w.x * s; b[n + 1] = w.y * s; b[n + 2] = w.z * s; b[n + 3] = w.w * s;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int n = 0; n < RN; ++n) acc[m][n] = fmaf(a[m], b[n], acc[m][n]);
  }
}

// Rows r < L of a [C][cols] block from a token-major workspace array (row r is
// token tok0 + r, `stride` floats apart) into shared rows `ld` floats apart;
// rows L..C-1 zero.  cols is a multiple of 4.  Issued as 16-byte cp.async
// copies (zero-filled past L), so all of a block is in flight at once; the
// caller waits with cp_async_wait_all() and a barrier.
__device__ __forceinline__ void load_rows(float* dst, int ld, const float* src, size_t stride,
                                          int C, int L, int cols) {
  const int c4 = cols / 4;
  for (int e = threadIdx.x; e < C * c4; e += blockDim.x) {
    const int r = e / c4, q = e % c4;
    const float* g = r < L ? src + (size_t)r * stride + 4 * q : src;   // src: not read when r >= L
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst + r * ld + 4 * q);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(g),
                 "r"(r < L ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---- the chunk-local WY factors: one CTA per (chunk, value head) ---------------
// Shared-memory layout (floats): K [C][DK+4] | Q, then V [C][max(DK+4, DV)] |
// AT [C][C+4] | gamma [C] | beta [C] | beta e^gamma [C].  AT holds A in its
// strict lower triangle and, once inverted, T transposed in its upper triangle
// and diagonal (T[r][j] at AT[j][r], j <= r): one C x C array instead of two,
// so that chunk 128 fits at head dim 128.
struct ChunkSmem {
  int K, QV, A, gam, beta, be, n;
  __host__ __device__ ChunkSmem(int C, int DK, int DV) {
    const int qv = (DK + 4) > DV ? DK + 4 : DV;
    int o = 0;
    K = o; o += C * (DK + 4);
    QV = o; o += C * qv;
    A = o; o += C * (C + 4);
    gam = o; o += C;
    beta = o; o += C;
    be = o; o += C;
    n = o;
  }
};

// Chunk x of the whole batch (chunk_off[b] <= x < chunk_off[b+1]) and value head
// h: with gamma the cumulative log-decay inside the chunk,
//   A = strict_tril(diag(beta) K K^T * e^{gamma_r - gamma_s}),  T = (I + A)^-1,
//   U = T diag(beta) V,  Wk = T diag(beta e^gamma) K,
//   P = tril(Q K^T * e^{gamma_r - gamma_s})
// written by token rows to ws_u, ws_wk, ws_p, with gamma to ws_gam.
__global__ void __launch_bounds__(256, 2) chunk_simt_kernel(const GdnPrefillArgs args) {
  extern __shared__ __align__(16) float sm[];
  if (!args.ws_flag[0]) return;
  const int x = blockIdx.x, h = blockIdx.y;
  const int B = args.num_seqs;
  if (x >= args.chunk_off[B]) return;
  int lo = 0, hi = B - 1;   // the largest b with chunk_off[b] <= x (skips empty sequences)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (args.chunk_off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int slot = args.slot_idx[b];
  if (slot < 0 || slot >= args.num_slots) return;   // status set by the scan
  const int C = args.chunk, DK = args.d_k, DV = args.d_v;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int64_t start = args.cu_seqlens[b];
  const int64_t Tlen = args.cu_seqlens[b + 1] - start;
  const int64_t c0 = (int64_t)(x - args.chunk_off[b]) * C;
  const int L = (Tlen - c0) < (int64_t)C ? (int)(Tlen - c0) : C;
  const int hk = h / (args.h_v / args.h_k);
  const int64_t tok0 = start + c0;

  const ChunkSmem S(C, DK, DV);
  const int KS = DK + 4, CS = C + 4, QS = (DK + 4) > DV ? DK + 4 : DV;
  float* sK = sm + S.K;
  float* sQV = sm + S.QV;
  float* sA = sm + S.A;   // A, then A below the diagonal and T^T on and above it
  float* sG = sm + S.gam;
  float* sB = sm + S.beta;
  float* sBe = sm + S.be;

  load_rows(sK, KS, args.ws_k + ((size_t)tok0 * args.h_k + hk) * DK, (size_t)args.h_k * DK, C, L, DK);
  load_rows(sQV, QS, args.ws_q + ((size_t)tok0 * args.h_k + hk) * DK, (size_t)args.h_k * DK, C, L, DK);
  if (tid < 32) {
    // cumulative log-decay over the chunk: a warp-wide scan per 32 rows
    float carry = 0.f;
    for (int r0 = 0; r0 < C; r0 += 32) {
      const int r = r0 + tid;
      float g = r < L ? args.ws_g[(size_t)(tok0 + r) * args.h_v + h] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, g, off);
        if (tid >= off) g += o;
      }
      g += carry;
      if (r < C) {
        sG[r] = g;
        sB[r] = r < L ? args.ws_beta[(size_t)(tok0 + r) * args.h_v + h] : 0.f;
      }
      carry = __shfl_sync(0xffffffffu, g, 31);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  for (int r = tid; r < C; r += NT) sBe[r] = sB[r] * expf(sG[r]);
  // A into shared memory, P straight to the workspace (rows r < L); a thread
  // takes rows ti + m C/4 and columns tj + n C/4
  const int nb = C / 4;
  for (int tile = tid; tile < nb * nb; tile += NT) {
    // a warp takes 4 row blocks x 8 column blocks (when nb allows): its eight
    // K rows per load step sit 4 (d_k + 4) floats apart, eight distinct banks
    int ti = tile / nb, tj = tile % nb;
    if (nb % 8 == 0) {
      const int blk = tile >> 5, ln = tile & 31, nbj = nb / 8;
      ti = 4 * (blk / nbj) + (ln >> 3);
      tj = 8 * (blk % nbj) + (ln & 7);
    }
    float a[4][4] = {}, p[4][4] = {};
    tile_rows_rows<4, 4>(a, sK, KS, ti, sK, KS, tj, nb, DK);
    tile_rows_rows<4, 4>(p, sQV, QS, ti, sK, KS, tj, nb, DK);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int r = ti + m * nb;
      float* prow = args.ws_p + ((size_t)(tok0 + r) * args.h_v + h) * C;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int s = tj + n * nb;
        const float dec = s <= r ? expf(sG[r] - sG[s]) : 0.f;   // exponent <= 0
        sA[r * CS + s] = s < r ? sB[r] * a[m][n] * dec : 0.f;
        if (r < L) prow[s] = p[m][n] * dec;
      }
    }
  }
  __syncthreads();
  // V over Q (Q is no longer read), in flight during the inverse
  load_rows(sQV, QS, args.ws_v + ((size_t)tok0 * args.h_v + h) * DV, (size_t)args.h_v * DV, C, L, DV);
  // T = (I + A)^-1 by forward substitution down each column j: T[r][j] =
  // delta_rj - sum_{j<=s<r} A[r][s] T[s][j] (T[s][j] = 0 for s < j).  TPC = NT / C
  // threads share a column (adjacent lanes); thread q of the group owns the
  // rows s = q mod TPC, sums its part of each row's series and the group adds
  // the parts with shuffles.  T[s][j] goes to AT[j][s] (on or above the
  // diagonal, where A is zero and never read); each is written and read only
  // by its owner.  Every lane runs every row (the shuffles are warp-wide).
  {
    const int TPC = NT / C;   // 2, 4, 8 or 16 (NT = 256, C = 128, 64, 32, 16)
    const int j = tid / TPC, q = tid % TPC;
    for (int r = 0; r < C; ++r) {
      float part = 0.f;
      for (int s2 = q; s2 < r; s2 += TPC)
        if (s2 >= j) part = fmaf(sA[r * CS + s2], sA[j * CS + s2], part);
      for (int m = TPC >> 1; m >= 1; m >>= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
      if (r % TPC == q && r >= j) sA[j * CS + r] = r == j ? 1.f : -part;
    }
  }
  cp_async_wait_all();
  __syncthreads();
  // U = T diag(beta) V and Wk = T diag(beta e^gamma) K, 4 x 8 blocks (the U
  // blocks first, then the Wk ones; consecutive blocks share their rows, so a
  // warp reads at most two rows of T at a time); T is lower triangular, so row
  // block r0 needs k < r0 + 4 only
  const int nv = DV / 8, nk = DK / 8;
  for (int tile = tid; tile < nb * (nv + nk); tile += NT) {
    const bool is_u = tile < nb * nv;
    const int t2 = is_u ? tile : tile - nb * nv;
    const int ncb = is_u ? nv : nk;
    const int r0 = (t2 / ncb) * 4;
    const int c0c = (t2 % ncb) * 8;
    float acc[4][8] = {};
    if (is_u) tile_tt_cols<8>(acc, sA, CS, r0, sQV, QS, c0c, sB);
    else tile_tt_cols<8>(acc, sA, CS, r0, sK, KS, c0c, sBe);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int r = r0 + m;
      if (r >= L) continue;
      float* dst = is_u ? args.ws_u + ((size_t)(tok0 + r) * args.h_v + h) * DV + c0c
                        : args.ws_wk + ((size_t)(tok0 + r) * args.h_v + h) * DK + c0c;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
    }
  }
  for (int r = tid; r < L; r += NT) args.ws_gam[(size_t)(tok0 + r) * args.h_v + h] = sG[r];
}

// ---- the scan: one CTA per (sequence, value head, d_v tile) --------------------
// Shared-memory layout (floats): S^T [DK][DVT] | Wk [C][DK+4] | Q [C][DK+4] |
// K [C][DK+4] | P [C][C+4] | U, then W [C][DVT] | e^gamma [C] | e^{gamma_last - gamma} [C].
struct ScanSmem {
  int H, Wk, Q, K, P, W, eg, dl, n;
  __host__ __device__ ScanSmem(int C, int DK, int DVT) {
    int o = 0;
    H = o; o += DK * DVT;
    Wk = o; o += C * (DK + 4);
    Q = o; o += C * (DK + 4);
    K = o; o += C * (DK + 4);
    P = o; o += C * (C + 4);
    W = o; o += C * DVT;
    eg = o; o += C;
    dl = o; o += C;
    n = o;
  }
};

// Per chunk, with the chunk's Wk, U, P and gamma from chunk_simt_kernel:
//   W = U - Wk S^T
//   O = diag(e^gamma) Q S^T + P W
//   S^T <- e^{gamma_last} S^T + K^T diag(e^{gamma_last - gamma}) W
// The state tile S^T [DK][DVT] stays in shared memory for the whole sequence.
// Register blocks: RMW x 4 for the [C][DVT] products, RMS x 4 for the state
// update (smaller blocks for narrow tiles keep every thread busy).
template <typename IO, int RMW, int RMS>
__global__ void __launch_bounds__(256) scan_simt_kernel(const GdnPrefillArgs args, int DVT) {
  extern __shared__ __align__(16) float sm[];
  if (!args.ws_flag[0]) return;
  const int b = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * DVT;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int C = args.chunk, DK = args.d_k, DV = args.d_v;
  const int slot = args.slot_idx[b];
  if (slot < 0 || slot >= args.num_slots) {
    if (h == 0 && blockIdx.z == 0 && tid == 0) set_status(args.d_status, GDN_DEV_BAD_SLOT);
    return;
  }
  const ScanSmem S(C, DK, DVT);
  const int KS = DK + 4, CS = C + 4;
  float* sH = sm + S.H;     // [DK][DVT]   S^T tile
  float* sWk = sm + S.Wk;   // [C][KS]
  float* sQ = sm + S.Q;     // [C][KS]
  float* sK = sm + S.K;     // [C][KS]
  float* sP = sm + S.P;     // [C][CS]
  float* sW = sm + S.W;     // [C][DVT]    U, then W
  float* sEg = sm + S.eg;   // [C]
  float* sDl = sm + S.dl;   // [C]

  const int hk = h / (args.h_v / args.h_k);
  const int64_t start = args.cu_seqlens[b];
  const int64_t Tlen = args.cu_seqlens[b + 1] - start;
  const bool init = args.has_init ? args.has_init[b] != 0 : false;
  float* gstate = args.state_pool + ((size_t)slot * args.h_v + h) * (size_t)DK * DV;
  for (int e = tid; e < DK * DVT; e += NT) {
    const int i = e / DVT, j = e % DVT;
    sH[e] = init ? gstate[(size_t)i * DV + j0 + j] : 0.f;
  }
  IO* out = reinterpret_cast<IO*>(args.o);
  const int nr = C / RMW, nc = DVT / 4;   // RMW x 4 blocks of the [C][DVT] products
  const int ni = DK / RMS;                // RMS x 4 blocks of the [DK][DVT] state update

  // Wk, Q and P of a chunk are fetched while the previous chunk still runs,
  // as soon as it has finished reading them; K and U at the chunk's start.
  auto len_at = [&](int64_t cc) { return (Tlen - cc) < (int64_t)C ? (int)(Tlen - cc) : C; };
  auto fetch_wk = [&](int64_t cc) {
    load_rows(sWk, KS, args.ws_wk + ((size_t)(start + cc) * args.h_v + h) * DK,
              (size_t)args.h_v * DK, C, len_at(cc), DK);
  };
  auto fetch_qp = [&](int64_t cc) {
    load_rows(sQ, KS, args.ws_q + ((size_t)(start + cc) * args.h_k + hk) * DK,
              (size_t)args.h_k * DK, C, len_at(cc), DK);
    load_rows(sP, CS, args.ws_p + ((size_t)(start + cc) * args.h_v + h) * C, (size_t)args.h_v * C,
              C, len_at(cc), C);
  };
  if (Tlen > 0) {
    fetch_wk(0);
    fetch_qp(0);
  }
  for (int64_t c0 = 0; c0 < Tlen; c0 += C) {
    const int L = len_at(c0);
    const int64_t tok0 = start + c0;
    const bool more = c0 + C < Tlen;
    __syncthreads();   // the previous chunk's reads of K, W and S^T are done
    load_rows(sK, KS, args.ws_k + ((size_t)tok0 * args.h_k + hk) * DK, (size_t)args.h_k * DK, C, L, DK);
    load_rows(sW, DVT, args.ws_u + ((size_t)tok0 * args.h_v + h) * DV + j0, (size_t)args.h_v * DV, C, L, DVT);
    const float glast = args.ws_gam[(size_t)(tok0 + L - 1) * args.h_v + h];
    for (int r = tid; r < C; r += NT) {
      const float g = r < L ? args.ws_gam[(size_t)(tok0 + r) * args.h_v + h] : 0.f;
      sEg[r] = r < L ? expf(g) : 0.f;
      sDl[r] = r < L ? expf(glast - g) : 0.f;   // exponent <= 0
    }
    cp_async_wait_all();
    __syncthreads();
    // W = U - Wk S^T (each block read and written by its own thread)
    for (int tile = tid; tile < nr * nc; tile += NT) {
      const int r0 = (tile / nc) * RMW, cc = (tile % nc) * 4;
      float acc[RMW][4] = {};
      tile_rows_cols<RMW, 4>(acc, sWk, KS, r0, sH, DVT, cc, 0, DK, nullptr);
#pragma unroll
      for (int m = 0; m < RMW; ++m) {
        float4* w = reinterpret_cast<float4*>(sW + (r0 + m) * DVT + cc);
        const float4 u = *w;
        *w = make_float4(u.x - acc[m][0], u.y - acc[m][1], u.z - acc[m][2], u.w - acc[m][3]);
      }
    }
    __syncthreads();
    if (more) fetch_wk(c0 + C);   // Wk is not read again in this chunk
    // O = diag(e^gamma) Q S^T + P W; P is lower triangular, so row block r0
    // needs W rows < r0 + RMW only
    for (int tile = tid; tile < nr * nc; tile += NT) {
      const int r0 = (tile / nc) * RMW, cc = (tile % nc) * 4;
      float acc[RMW][4] = {};
      tile_rows_cols<RMW, 4>(acc, sQ, KS, r0, sH, DVT, cc, 0, DK, nullptr);
#pragma unroll
      for (int m = 0; m < RMW; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[m][n] *= sEg[r0 + m];
      tile_rows_cols<RMW, 4>(acc, sP, CS, r0, sW, DVT, cc, 0, r0 + RMW, nullptr);
#pragma unroll
      for (int m = 0; m < RMW; ++m) {
        const int r = r0 + m;
        if (r >= L) continue;
        IO* orow = out + ((size_t)(tok0 + r) * args.h_v + h) * DV + j0 + cc;
#pragma unroll
        for (int n = 0; n < 4; ++n) st_io(orow + n, acc[m][n]);
      }
    }
    __syncthreads();
    if (more) fetch_qp(c0 + C);   // nor are Q and P
    // S^T <- e^{gamma_last} S^T + K^T diag(e^{gamma_last - gamma}) W, 8 x 4
    // blocks (rows of K beyond the chunk's end are zero, their weight too)
    const float dlast = expf(glast);
    // interval checkpoint: the state after these c0 / C + 1 chunks, each thread
    // storing the elements it just updated
    const int64_t cs = args.ckpt_every_chunks > 0 ? ckpt_slot_of(args, b, c0 / C + 1, Tlen) : -1;
    float* cst = cs >= 0 ? args.state_pool + ((size_t)cs * args.h_v + h) * (size_t)DK * DV : nullptr;
    for (int tile = tid; tile < ni * nc; tile += NT) {
      const int i0 = (tile / nc) * RMS, cc = (tile % nc) * 4;
      float acc[RMS][4] = {};
      tile_cols_cols<RMS, 4>(acc, sK, KS, i0, sW, DVT, cc, L, sDl);
#pragma unroll
      for (int m = 0; m < RMS; ++m) {
        float4* hp = reinterpret_cast<float4*>(sH + (i0 + m) * DVT + cc);
        const float4 o = *hp;
        const float4 nv = make_float4(fmaf(dlast, o.x, acc[m][0]), fmaf(dlast, o.y, acc[m][1]),
                                      fmaf(dlast, o.z, acc[m][2]), fmaf(dlast, o.w, acc[m][3]));
        *hp = nv;
        if (cst) *reinterpret_cast<float4*>(cst + (size_t)(i0 + m) * DV + j0 + cc) = nv;
      }
    }
  }
  cp_async_wait_all();   // nothing in flight (the last chunk fetched nothing ahead)
  __syncthreads();
  for (int e = tid; e < DK * DVT; e += NT) {
    const int i = e / DVT, j = e % DVT;
    gstate[(size_t)i * DV + j0 + j] = sH[e];
  }
}

// ---- the scan with its chunk inputs streamed through two buffers ------------
// For chunks whose Wk, Q and K rows do not fit in shared memory side by side
// (chunk 128 at head dim 128): the three [C][DK+4] blocks of a chunk pass
// through two buffers in the order they are used (Wk, Q, K, next Wk, ...), each
// fetched while the previous one is in use.  Shared-memory layout (floats):
// S^T [DK][DVT] | X0, X1 [C][DK+4] | P [C][C+4] | U, then W [C][DVT] |
// e^gamma [C] | e^{gamma_last - gamma} [C].  Same arithmetic as scan_simt_kernel.
struct ScanStreamSmem {
  int H, X0, X1, P, W, eg, dl, n;
  __host__ __device__ ScanStreamSmem(int C, int DK, int DVT) {
    int o = 0;
    H = o; o += DK * DVT;
    X0 = o; o += C * (DK + 4);
    X1 = o; o += C * (DK + 4);
    P = o; o += C * (C + 4);
    W = o; o += C * DVT;
    eg = o; o += C;
    dl = o; o += C;
    n = o;
  }
};

template <typename IO, int RMW, int RMS>
__global__ void __launch_bounds__(256) scan_simt_stream_kernel(const GdnPrefillArgs args, int DVT) {
  extern __shared__ __align__(16) float sm[];
  if (!args.ws_flag[0]) return;
  const int b = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * DVT;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int C = args.chunk, DK = args.d_k, DV = args.d_v;
  const int slot = args.slot_idx[b];
  if (slot < 0 || slot >= args.num_slots) {
    if (h == 0 && blockIdx.z == 0 && tid == 0) set_status(args.d_status, GDN_DEV_BAD_SLOT);
    return;
  }
  const ScanStreamSmem S(C, DK, DVT);
  const int KS = DK + 4, CS = C + 4;
  float* sH = sm + S.H;
  float* const sX0 = sm + S.X0;
  float* const sX1 = sm + S.X1;
  float* sP = sm + S.P;
  float* sW = sm + S.W;
  float* sEg = sm + S.eg;
  float* sDl = sm + S.dl;

  const int hk = h / (args.h_v / args.h_k);
  const int64_t start = args.cu_seqlens[b];
  const int64_t Tlen = args.cu_seqlens[b + 1] - start;
  const bool init = args.has_init ? args.has_init[b] != 0 : false;
  float* gstate = args.state_pool + ((size_t)slot * args.h_v + h) * (size_t)DK * DV;
  for (int e = tid; e < DK * DVT; e += NT) {
    const int i = e / DVT, j = e % DVT;
    sH[e] = init ? gstate[(size_t)i * DV + j0 + j] : 0.f;
  }
  IO* out = reinterpret_cast<IO*>(args.o);
  const int nr = C / RMW, nc = DVT / 4;
  const int ni = DK / RMS;
  auto len_at = [&](int64_t cc) { return (Tlen - cc) < (int64_t)C ? (int)(Tlen - cc) : C; };
  // block i of the stream (3 per chunk: Wk, Q, K) goes to buffer i % 2
  auto fetch = [&](int64_t cc, int which, float* dst) {
    const int L = len_at(cc);
    if (which == 0)
      load_rows(dst, KS, args.ws_wk + ((size_t)(start + cc) * args.h_v + h) * DK,
                (size_t)args.h_v * DK, C, L, DK);
    else
      load_rows(dst, KS, (which == 1 ? args.ws_q : args.ws_k) + ((size_t)(start + cc) * args.h_k + hk) * DK,
                (size_t)args.h_k * DK, C, L, DK);
  };
  auto fetch_p = [&](int64_t cc) {
    load_rows(sP, CS, args.ws_p + ((size_t)(start + cc) * args.h_v + h) * C, (size_t)args.h_v * C, C,
              len_at(cc), C);
  };
  int64_t blk = 0;   // stream index of the chunk's Wk block
  if (Tlen > 0) {
    fetch(0, 0, sX0);
    fetch_p(0);
  }
  for (int64_t c0 = 0; c0 < Tlen; c0 += C, blk += 3) {
    const int L = len_at(c0);
    const int64_t tok0 = start + c0;
    const bool more = c0 + C < Tlen;
    float* const xWk = (blk & 1) ? sX1 : sX0;   // the K block reuses this buffer
    float* const xQ = (blk & 1) ? sX0 : sX1;
    __syncthreads();   // the previous chunk's reads of its K block, W and S^T are done
    load_rows(sW, DVT, args.ws_u + ((size_t)tok0 * args.h_v + h) * DV + j0, (size_t)args.h_v * DV, C, L, DVT);
    fetch(c0, 1, xQ);
    const float glast = args.ws_gam[(size_t)(tok0 + L - 1) * args.h_v + h];
    for (int r = tid; r < C; r += NT) {
      const float g = r < L ? args.ws_gam[(size_t)(tok0 + r) * args.h_v + h] : 0.f;
      sEg[r] = r < L ? expf(g) : 0.f;
      sDl[r] = r < L ? expf(glast - g) : 0.f;   // exponent <= 0
    }
    asm volatile("cp.async.wait_group 1;" ::: "memory");   // Wk, P and U (Q may still fly)
    __syncthreads();
    // W = U - Wk S^T
    for (int tile = tid; tile < nr * nc; tile += NT) {
      const int r0 = (tile / nc) * RMW, cc = (tile % nc) * 4;
      float acc[RMW][4] = {};
      tile_rows_cols<RMW, 4>(acc, xWk, KS, r0, sH, DVT, cc, 0, DK, nullptr);
#pragma unroll
      for (int m = 0; m < RMW; ++m) {
        float4* w = reinterpret_cast<float4*>(sW + (r0 + m) * DVT + cc);
        const float4 u = *w;
        *w = make_float4(u.x - acc[m][0], u.y - acc[m][1], u.z - acc[m][2], u.w - acc[m][3]);
      }
    }
    __syncthreads();
    float* const xK = xWk;
    fetch(c0, 2, xK);   // into the Wk block's buffer
    asm volatile("cp.async.wait_group 1;" ::: "memory");   // Q (K may still fly)
    __syncthreads();
    // O = diag(e^gamma) Q S^T + P W
    for (int tile = tid; tile < nr * nc; tile += NT) {
      const int r0 = (tile / nc) * RMW, cc = (tile % nc) * 4;
      float acc[RMW][4] = {};
      tile_rows_cols<RMW, 4>(acc, xQ, KS, r0, sH, DVT, cc, 0, DK, nullptr);
#pragma unroll
      for (int m = 0; m < RMW; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[m][n] *= sEg[r0 + m];
      tile_rows_cols<RMW, 4>(acc, sP, CS, r0, sW, DVT, cc, 0, r0 + RMW, nullptr);
#pragma unroll
      for (int m = 0; m < RMW; ++m) {
        const int r = r0 + m;
        if (r >= L) continue;
        IO* orow = out + ((size_t)(tok0 + r) * args.h_v + h) * DV + j0 + cc;
#pragma unroll
        for (int n = 0; n < 4; ++n) st_io(orow + n, acc[m][n]);
      }
    }
    __syncthreads();
    if (more) {   // the next chunk's Wk into the Q block's buffer, its P
      fetch(c0 + C, 0, xQ);
      fetch_p(c0 + C);
      asm volatile("cp.async.wait_group 2;" ::: "memory");   // K
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    // S^T <- e^{gamma_last} S^T + K^T diag(e^{gamma_last - gamma}) W
    const float dlast = expf(glast);
    const int64_t cs = args.ckpt_every_chunks > 0 ? ckpt_slot_of(args, b, c0 / C + 1, Tlen) : -1;
    float* cst = cs >= 0 ? args.state_pool + ((size_t)cs * args.h_v + h) * (size_t)DK * DV : nullptr;
    for (int tile = tid; tile < ni * nc; tile += NT) {
      const int i0 = (tile / nc) * RMS, cc = (tile % nc) * 4;
      float acc[RMS][4] = {};
      tile_cols_cols<RMS, 4>(acc, xK, KS, i0, sW, DVT, cc, L, sDl);
#pragma unroll
      for (int m = 0; m < RMS; ++m) {
        float4* hp = reinterpret_cast<float4*>(sH + (i0 + m) * DVT + cc);
        const float4 o = *hp;
        const float4 nv = make_float4(fmaf(dlast, o.x, acc[m][0]), fmaf(dlast, o.y, acc[m][1]),
                                      fmaf(dlast, o.z, acc[m][2]), fmaf(dlast, o.w, acc[m][3]));
        *hp = nv;
        if (cst) *reinterpret_cast<float4*>(cst + (size_t)(i0 + m) * DV + j0 + cc) = nv;
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  for (int e = tid; e < DK * DVT; e += NT) {
    const int i = e / DVT, j = e % DVT;
    gstate[(size_t)i * DV + j0 + j] = sH[e];
  }
}

// d_v tile of the scan: 64 wide, or 32 when 64-wide tiles would leave SMs idle
// (fewer (sequence, head, tile) CTAs than SMs); sms <= 0: the largest tile.
static int scan_dv_tile(int d_v, int64_t seq_heads = 0, int sms = 0) {
  if (d_v < 64) return d_v;
  if (sms > 0 && seq_heads * (d_v / 64) < sms) return 32;
  return 64;
}

// The scan's plan: the d_v tile and whether the chunk inputs stream through two
// buffers (when Wk, Q and K side by side do not fit in shared memory), with its
// shared-memory bytes.  A plan above the limit is rejected by the caller.
constexpr size_t kScanSmemLimit = 227 * 1024;
struct ScanPlan {
  int dvt;
  bool stream;
  size_t bytes;
};
static ScanPlan scan_plan(int C, int DK, int DV, int64_t seq_heads = 0, int sms = 0) {
  const int dvt = scan_dv_tile(DV, seq_heads, sms);
  const size_t std_bytes = (size_t)ScanSmem(C, DK, dvt).n * sizeof(float);
  if (std_bytes <= kScanSmemLimit) return {dvt, false, std_bytes};
  for (int t = dvt; t >= 8; t /= 2) {
    const size_t b = (size_t)ScanStreamSmem(C, DK, t).n * sizeof(float);
    if (b <= kScanSmemLimit) return {t, true, b};
  }
  return {dvt, false, std_bytes};
}

static int num_sms() {
  static int n = 0;   // the device's SM count, looked up once per process
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 0;
  }
  return n;
}

template <typename IO>
static cudaError_t launch_simt(const GdnPrefillArgs& a, cudaStream_t s, gdn_trace* tr) {
  cudaError_t e = gdn_trace_mark(tr, 0, true, s);
  if (e != cudaSuccess) return e;
  check_cu_seqlens_kernel<<<1, 256, 0, s>>>(a.cu_seqlens, a.num_seqs, a.total_tokens, a.chunk,
                                            a.chunk_off, a.ws_flag, a.d_status);
  gdn_trace_count(tr, 1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.total_tokens > 0) {
    const size_t fe_smem = (size_t)a.conv_dim * sizeof(float);
    if (fe_smem > 48 * 1024) {
      e = cudaFuncSetAttribute(frontend_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)fe_smem);
      if (e != cudaSuccess) return e;
    }
    frontend_kernel<IO><<<(unsigned)a.total_tokens, 256, fe_smem, s>>>(a);
    gdn_trace_count(tr, 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e = gdn_launch_window(a, std::is_same<IO, float>::value ? GDN_FP32 : GDN_BF16, s, tr);
  if (e != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 0, false, s)) != cudaSuccess) return e;
  if (a.total_tokens > 0) {
    if ((e = gdn_trace_mark(tr, 1, true, s)) != cudaSuccess) return e;
    const size_t csmem = (size_t)ChunkSmem(a.chunk, a.d_k, a.d_v).n * sizeof(float);
    e = cudaFuncSetAttribute(chunk_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)csmem);
    if (e != cudaSuccess) return e;
    dim3 cgrid((unsigned)a.max_chunks, a.h_v);
    chunk_simt_kernel<<<cgrid, 256, csmem, s>>>(a);
    gdn_trace_count(tr, 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if ((e = gdn_trace_mark(tr, 1, false, s)) != cudaSuccess) return e;
  }
  const ScanPlan plan = scan_plan(a.chunk, a.d_k, a.d_v, (int64_t)a.num_seqs * a.h_v, num_sms());
  const int DVT = plan.dvt;
  const size_t smem = plan.bytes;
  // 32-wide (or narrower) tiles: 2 x 4 and 4 x 4 blocks, else 4 x 4 and 8 x 4
  auto kern = plan.stream ? (DVT <= 32 ? scan_simt_stream_kernel<IO, 2, 4> : scan_simt_stream_kernel<IO, 4, 8>)
                          : (DVT == 32 ? scan_simt_kernel<IO, 2, 4> : scan_simt_kernel<IO, 4, 8>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 2, true, s)) != cudaSuccess) return e;
  dim3 grid(a.num_seqs, a.h_v, a.d_v / DVT);
  kern<<<grid, 256, smem, s>>>(a, DVT);
  gdn_trace_count(tr, 1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return gdn_trace_mark(tr, 2, false, s);
}

}  // namespace gdn

cudaError_t gdn_launch_check(const GdnPrefillArgs& a, cudaStream_t s, gdn_trace* tr) {
  gdn::check_cu_seqlens_kernel<<<1, 256, 0, s>>>(a.cu_seqlens, a.num_seqs, a.total_tokens,
                                                 a.chunk, nullptr, a.ws_flag, a.d_status);
  gdn_trace_count(tr, 1);
  return cudaGetLastError();
}

cudaError_t gdn_launch_window(const GdnPrefillArgs& a, int io, cudaStream_t s, gdn_trace* tr) {
  // z = 0: each sequence's own window; z >= 1: its interval checkpoints (each
  // z-block loops over every (gridDim.z - 1)-th one), as many z-blocks as a
  // sequence of average length has checkpoints, 1 to 64
  int64_t nz = 1;
  if (a.ckpt_every_chunks > 0) {
    const int64_t every = (int64_t)a.ckpt_every_chunks * a.chunk;
    const int64_t avg = (a.total_tokens / (a.num_seqs > 0 ? a.num_seqs : 1) + every - 1) / every;
    nz = 1 + (avg < 1 ? 1 : (avg > 64 ? 64 : avg));
  }
  dim3 wgrid(a.num_seqs, (a.conv_dim + 255) / 256, (unsigned)nz);
  if (io == GDN_BF16)
    gdn::window_writeback_kernel<__nv_bfloat16><<<wgrid, 256, 0, s>>>(a);
  else
    gdn::window_writeback_kernel<float><<<wgrid, 256, 0, s>>>(a);
  gdn_trace_count(tr, 1);
  return cudaGetLastError();
}

size_t gdn_simt_scan_smem_bytes(int chunk, int d_k, int d_v) {
  const size_t scan = gdn::scan_plan(chunk, d_k, d_v).bytes;
  const size_t chk = (size_t)gdn::ChunkSmem(chunk, d_k, d_v).n * sizeof(float);
  return scan > chk ? scan : chk;
}

cudaError_t gdn_launch_prefill_simt(const GdnPrefillArgs& a, int io, cudaStream_t s,
                                    gdn_trace* tr) {
  if (a.num_seqs == 0) return cudaSuccess;
  return io == GDN_BF16 ? gdn::launch_simt<__nv_bfloat16>(a, s, tr)
                        : gdn::launch_simt<float>(a, s, tr);
}
