// gdn_prefill_simt.cu -- chunked prefill of the Gated DeltaNet layer on the
// fp32 SIMT pipes, for every supported shape (d_k, d_v in {16,32,64,128},
// chunk in {16,32,64}, fp32 or bf16 I/O).  The tensor-core path takes the
// Qwen3.5-4B layer shape; this path serves the other shapes and fp32 I/O, whose
// 1e-3 tolerance bf16 tensor-core operands would not meet.
//
// Kernels, in stream order:
//   1. check_cu_seqlens   one CTA; sets the workspace flag (and the device
//                         status bit when cu_seqlens is malformed).
//   2. frontend           one CTA per token: causal conv (window or zero
//                         history before the sequence start) + SiLU, L2 norm
//                         of q and k with the 1/sqrt(d_k) query scale, gates.
//   3. window_writeback   the last W-1 raw inputs of each sequence to its slot.
//   4. scan               one CTA per (sequence, value head, d_v tile): the
//                         chunked WY form, sequential over chunks, state in
//                         shared memory.  Per chunk with cumulative log-decay
//                         gamma (oxydllm 0.0.0-alpha.12.2 release notes, New
//                         Features, "Gated DeltaNet runtime": chunked parallel
//                         scan, per-chunk unit-lower-triangular system):
//       A = strict_tril(diag(beta) K K^T * e^{gamma_r - gamma_s})
//       T = (I + A)^-1           (column-wise forward substitution: exact
//                                 entries, no matrix powers, finite on fully
//                                 correlated keys)
//       U = T diag(beta) V,  Wk = T diag(beta e^gamma) K
//       W = U - Wk S^T
//       O = diag(e^gamma) Q S^T + tril(Q K^T * e^{gamma_r - gamma_s}) W
//       S^T <- e^{gamma_last} S^T + K^T diag(e^{gamma_last - gamma}) W
//     Only e^{x} with x <= 0 is ever formed.
#include <type_traits>

#include "gdn_common.cuh"

namespace gdn {

__global__ void check_cu_seqlens_kernel(const int32_t* __restrict__ cu, int num_seqs,
                                        int64_t total, int32_t* flag, int32_t* d_status) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = (cu[0] != 0) || ((int64_t)cu[num_seqs] != total);
  __syncthreads();
  for (int i = threadIdx.x; i < num_seqs; i += blockDim.x)
    if (cu[i + 1] < cu[i]) bad = 1;
  __syncthreads();
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

  for (int c = threadIdx.x; c < cd; c += blockDim.x) {
    const float4 w = *reinterpret_cast<const float4*>(args.conv_weight + 4 * (size_t)c);
    const float wt[4] = {w.x, w.y, w.z, w.w};
    float z = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t tau = p - 3 + k;  // position of this tap's input
      float xv;
      if (tau >= 0) xv = ld_io(x + (size_t)(tok - 3 + k) * cd + c);
      else xv = init ? ld_io(win + (size_t)(3 + tau) * cd + c) : 0.f;
      z = fmaf(wt[k], xv, z);
    }
    s_y[c] = silu(z);
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

struct ScanSmem {
  // offsets in floats; K and Q rows are padded to d_k + 1 floats, so that the
  // lanes of a warp reading one column of K for different tokens (K K^T, Q K^T)
  // hit different banks
  int H, K, Q, V, U, Wk, A, T, gam, beta, be, dl, eg, n;
  __host__ __device__ ScanSmem(int C, int DK, int DVT) {
    int o = 0;
    H = o; o += DK * DVT;
    K = o; o += C * (DK + 1);
    Q = o; o += C * (DK + 1);
    V = o; o += C * DVT;
    U = o; o += C * DVT;
    Wk = o; o += C * DK;
    A = o; o += C * C;
    T = o; o += C * C;
    gam = o; o += C;
    beta = o; o += C;
    be = o; o += C;   // beta_s e^{gamma_s}
    dl = o; o += C;   // e^{gamma_last - gamma_r}
    eg = o; o += C;   // e^{gamma_r}
    n = o;
  }
};

template <typename IO>
__global__ void __launch_bounds__(256) scan_simt_kernel(const GdnPrefillArgs args, int DVT) {
  extern __shared__ float sm[];
  if (!args.ws_flag[0]) return;
  const int b = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * DVT;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int C = args.chunk, DK = args.d_k, DV = args.d_v;
  const int slot = args.slot_idx[b];
  if (slot < 0 || slot >= args.num_slots) {
    if (h == 0 && blockIdx.z == 0 && tid == 0 && slot >= args.num_slots)
      set_status(args.d_status, GDN_DEV_BAD_SLOT);
    return;
  }
  const ScanSmem L(C, DK, DVT);
  float* sH = sm + L.H;    // [DK][DVT]   S^T tile
  float* sK = sm + L.K;    // [C][DK + 1]
  float* sQ = sm + L.Q;    // [C][DK + 1]
  float* sV = sm + L.V;    // [C][DVT]
  float* sU = sm + L.U;    // [C][DVT]    U, then W
  float* sWk = sm + L.Wk;  // [C][DK]
  float* sA = sm + L.A;    // [C][C]      A, then P
  float* sT = sm + L.T;    // [C][C]
  float* sG = sm + L.gam;  // [C]         cumulative log-decay
  float* sB = sm + L.beta; // [C]
  float* sBe = sm + L.be;  // [C]
  float* sDl = sm + L.dl;  // [C]
  float* sEg = sm + L.eg;  // [C]
  const int KS = DK + 1;   // row stride of sK, sQ

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

  for (int64_t c0 = 0; c0 < Tlen; c0 += C) {
    const int Lc = (Tlen - c0) < (int64_t)C ? (int)(Tlen - c0) : C;
    __syncthreads();
    for (int e = tid; e < C * DK; e += NT) {
      const int r = e / DK, i = e % DK;
      const size_t tk = (size_t)(start + c0 + r);
      sK[r * KS + i] = r < Lc ? args.ws_k[(tk * args.h_k + hk) * DK + i] : 0.f;
      sQ[r * KS + i] = r < Lc ? args.ws_q[(tk * args.h_k + hk) * DK + i] : 0.f;
    }
    for (int e = tid; e < C * DVT; e += NT) {
      const int r = e / DVT, j = e % DVT;
      const size_t tk = (size_t)(start + c0 + r);
      sV[e] = r < Lc ? args.ws_v[(tk * args.h_v + h) * DV + j0 + j] : 0.f;
    }
    if (tid == 0) {
      float acc = 0.f;
      for (int r = 0; r < C; ++r) {
        const size_t tk = (size_t)(start + c0 + r);
        acc += r < Lc ? args.ws_g[tk * args.h_v + h] : 0.f;
        sG[r] = acc;
        sB[r] = r < Lc ? args.ws_beta[tk * args.h_v + h] : 0.f;
      }
    }
    __syncthreads();
    for (int r = tid; r < C; r += NT) {
      sBe[r] = sB[r] * expf(sG[r]);
      sDl[r] = expf(sG[C - 1] - sG[r]);
      sEg[r] = expf(sG[r]);
    }
    // A (strictly lower), P (lower incl. diagonal) need K K^T and Q K^T
    for (int e = tid; e < C * C; e += NT) {
      const int r = e / C, s = e % C;
      float a = 0.f;
      if (s < r) {
        float dot = 0.f;
        for (int i = 0; i < DK; ++i) dot = fmaf(sK[r * KS + i], sK[s * KS + i], dot);
        a = sB[r] * dot * expf(sG[r] - sG[s]);
      }
      sA[e] = a;
    }
    __syncthreads();
    // T = (I + A)^-1 by forward substitution down each column j: T[r][j] =
    // delta_rj - sum_{s<r} A[r][s] T[s][j].  TPC = NT / C threads share a column
    // (adjacent lanes); thread q of the group owns the rows s = q mod TPC,
    // sums its part of each row's series and the group adds the parts with
    // shuffles.  Each T[s][j] is written and read only by its owner.
    {
      const int TPC = NT / C;              // 4, 8 or 16 (NT = 256, C = 64, 32, 16)
      const int j = tid / TPC, q = tid % TPC;
      for (int r = 0; r < C; ++r) {
        float part = 0.f;
        for (int s2 = q; s2 < r; s2 += TPC) part = fmaf(sA[r * C + s2], sT[s2 * C + j], part);
        for (int m = TPC >> 1; m >= 1; m >>= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
        if (r % TPC == q) sT[r * C + j] = r < j ? 0.f : (r == j ? 1.f : -part);
      }
    }
    __syncthreads();
    // U = T diag(beta) V ; Wk = T diag(beta e^gamma) K ; P -> sA
    for (int e = tid; e < C * DVT; e += NT) {
      const int r = e / DVT, j = e % DVT;
      float acc = 0.f;
      for (int s = 0; s <= r; ++s) acc = fmaf(sT[r * C + s] * sB[s], sV[s * DVT + j], acc);
      sU[e] = acc;
    }
    for (int e = tid; e < C * DK; e += NT) {
      const int r = e / DK, i = e % DK;
      float acc = 0.f;
      for (int s = 0; s <= r; ++s) acc = fmaf(sT[r * C + s] * sBe[s], sK[s * KS + i], acc);
      sWk[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < C * C; e += NT) {
      const int r = e / C, s = e % C;
      float p = 0.f;
      if (s <= r) {
        float dot = 0.f;
        for (int i = 0; i < DK; ++i) dot = fmaf(sQ[r * KS + i], sK[s * KS + i], dot);
        p = dot * expf(sG[r] - sG[s]);
      }
      sA[e] = p;
    }
    // W = U - Wk S^T  (in place in sU; each element read and written by one thread)
    for (int e = tid; e < C * DVT; e += NT) {
      const int r = e / DVT, j = e % DVT;
      float acc = 0.f;
      for (int i = 0; i < DK; ++i) acc = fmaf(sWk[r * DK + i], sH[i * DVT + j], acc);
      sU[e] -= acc;
    }
    __syncthreads();
    // O = diag(e^gamma) Q S^T + P W
    for (int e = tid; e < Lc * DVT; e += NT) {
      const int r = e / DVT, j = e % DVT;
      float qs = 0.f;
      for (int i = 0; i < DK; ++i) qs = fmaf(sQ[r * KS + i], sH[i * DVT + j], qs);
      float pw = 0.f;
      for (int s = 0; s <= r; ++s) pw = fmaf(sA[r * C + s], sU[s * DVT + j], pw);
      const float ov = fmaf(sEg[r], qs, pw);
      st_io(out + ((size_t)(start + c0 + r) * args.h_v + h) * DV + j0 + j, ov);
    }
    __syncthreads();
    // S^T <- e^{gamma_last} S^T + K^T diag(e^{gamma_last - gamma}) W
    const float glast = sG[C - 1];
    const float dlast = expf(glast);
    // interval checkpoint: the state after these c0 / C + 1 chunks, each thread
    // storing the elements it just updated
    const int64_t cs = args.ckpt_every_chunks > 0 ? ckpt_slot_of(args, b, c0 / C + 1, Tlen) : -1;
    float* cst = cs >= 0 ? args.state_pool + ((size_t)cs * args.h_v + h) * (size_t)DK * DV : nullptr;
    for (int e = tid; e < DK * DVT; e += NT) {
      const int i = e / DVT, j = e % DVT;
      float acc = 0.f;
      for (int r = 0; r < Lc; ++r) acc = fmaf(sK[r * KS + i] * sDl[r], sU[r * DVT + j], acc);
      sH[e] = fmaf(dlast, sH[e], acc);
      if (cst) cst[(size_t)i * DV + j0 + j] = sH[e];
    }
  }
  __syncthreads();
  for (int e = tid; e < DK * DVT; e += NT) {
    const int i = e / DVT, j = e % DVT;
    gstate[(size_t)i * DV + j0 + j] = sH[e];
  }
}

static int scan_dv_tile(int d_v) { return d_v < 64 ? d_v : 64; }

template <typename IO>
static cudaError_t launch_simt(const GdnPrefillArgs& a, cudaStream_t s, gdn_trace* tr) {
  cudaError_t e = gdn_trace_mark(tr, 0, true, s);
  if (e != cudaSuccess) return e;
  check_cu_seqlens_kernel<<<1, 256, 0, s>>>(a.cu_seqlens, a.num_seqs, a.total_tokens,
                                            a.ws_flag, a.d_status);
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
  const int DVT = scan_dv_tile(a.d_v);
  const ScanSmem L(a.chunk, a.d_k, DVT);
  const size_t smem = (size_t)L.n * sizeof(float);
  e = cudaFuncSetAttribute(scan_simt_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 2, true, s)) != cudaSuccess) return e;
  dim3 grid(a.num_seqs, a.h_v, a.d_v / DVT);
  scan_simt_kernel<IO><<<grid, 256, smem, s>>>(a, DVT);
  gdn_trace_count(tr, 1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return gdn_trace_mark(tr, 2, false, s);
}

}  // namespace gdn

cudaError_t gdn_launch_check(const GdnPrefillArgs& a, cudaStream_t s, gdn_trace* tr) {
  gdn::check_cu_seqlens_kernel<<<1, 256, 0, s>>>(a.cu_seqlens, a.num_seqs, a.total_tokens,
                                                 a.ws_flag, a.d_status);
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
  return (size_t)gdn::ScanSmem(chunk, d_k, gdn::scan_dv_tile(d_v)).n * sizeof(float);
}

cudaError_t gdn_launch_prefill_simt(const GdnPrefillArgs& a, int io, cudaStream_t s,
                                    gdn_trace* tr) {
  if (a.num_seqs == 0) return cudaSuccess;
  return io == GDN_BF16 ? gdn::launch_simt<__nv_bfloat16>(a, s, tr)
                        : gdn::launch_simt<float>(a, s, tr);
}
