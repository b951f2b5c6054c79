// gdn_decode.cu -- decode-time kernels of the Gated DeltaNet layer.
//
// gdn_decode_step: one token per row, O(1) in sequence length (oxydllm
// 0.0.0-alpha.12.2 release notes, New Features, "Gated DeltaNet runtime": the
// recurrent step for decode over the slot's conv window and F32 memory).
// One CTA per (row, key head) handles the H_v/H_k value heads that share the
// key head, so every conv-window channel it rolls belongs to exactly one CTA.
// Per value head the fp32 state (d_k x d_v, stored S^T, value index
// contiguous) is streamed through registers once: 128-bit evict-first loads,
// the two reductions u = S k^ and r = S q^ (in-thread over rows, then across
// warps through shared memory), then the rank-1 update written back with
// 128-bit evict-first stores.  The identity used:
//   S' = a S + b (v - a S k) k^T  =>  S'^T[i][j] = a S^T[i][j] + k_i d_j,
//   d_j = b (v_j - a u_j),  o_j = (S' q)_j = a r_j + d_j (k . q).
#include "gdn_common.cuh"

namespace gdn {

template <int DK, int DV>
struct DecodeCfg {
  static constexpr int NF4 = DK * DV / 4;  // float4 elements in one head's state
  static constexpr int NT = NF4 >= 1024 ? 256 : (NF4 >= 256 ? NF4 / 4 : (NF4 >= 32 ? NF4 : 32));
  static constexpr int F = NF4 / NT;       // float4 per thread
  static constexpr int CG = DV / 4;        // float4 column groups per state row
  static constexpr int RS = NT / CG;       // state rows covered by one sweep of the block
  static constexpr int NW = NT / 32;
  static_assert(NF4 % NT == 0 && NT % CG == 0 && F * RS == DK, "decode tiling");
};

// Causal width-4 conv of channel c for one decode token, plus the window roll.
// hist = (win[0][c], win[1][c], win[2][c], x[c]) oldest first; the window then
// becomes (win[1][c], win[2][c], x[c]).  Returns SiLU of the conv.
template <typename IO>
__device__ __forceinline__ float conv_step(int c, int conv_dim, const IO* __restrict__ xrow,
                                           IO* __restrict__ win,
                                           const float* __restrict__ conv_weight) {
  const float4 w = *reinterpret_cast<const float4*>(conv_weight + 4 * (size_t)c);
  const IO h0 = win[c];
  const IO h1 = win[conv_dim + c];
  const IO h2 = win[2 * (size_t)conv_dim + c];
  const IO xc = xrow[c];
  float z = w.x * ld_io(&h0);
  z = fmaf(w.y, ld_io(&h1), z);
  z = fmaf(w.z, ld_io(&h2), z);
  z = fmaf(w.w, ld_io(&xc), z);
  win[c] = h1;
  win[conv_dim + c] = h2;
  win[2 * (size_t)conv_dim + c] = xc;
  return silu(z);
}

template <int DK, int DV, typename IO>
__global__ void __launch_bounds__(DecodeCfg<DK, DV>::NT)
decode_step_kernel(const GdnDecodeArgs args) {
  using C = DecodeCfg<DK, DV>;
  const int n = blockIdx.x;
  const int hk = blockIdx.y;
  const int t = threadIdx.x;
  const int G = args.h_v / args.h_k;
  const int cd = args.conv_dim;
  IO* __restrict__ o = reinterpret_cast<IO*>(args.o);

  __shared__ float s_q[DK], s_k[DK], s_v[DV];
  __shared__ __align__(16) float s_delta[DV];
  __shared__ float s_red[2][C::NW][DV];
  __shared__ float s_scal[4];
  __shared__ float s_nrm[(DV + 31) / 32];   // fused gated norm: per-warp sums of o^2
  static_assert(C::NT >= DV, "one output value per thread");
  const bool fuse = args.z != nullptr;

  const int slot = args.slot_idx[n];
  if (slot < 0 || slot >= args.num_slots) {
    if (slot >= args.num_slots && t == 0) set_status(args.d_status, GDN_DEV_BAD_SLOT);
    for (int e = t; e < G * DV; e += C::NT) {
      const int h = hk * G + e / DV;
      st_io(o + ((size_t)n * args.h_v + h) * DV + (e % DV), 0.0f);
    }
    return;
  }

  const int cg = t % C::CG;   // columns 4cg .. 4cg+3
  const int r0 = t / C::CG;   // rows r0 + m*RS
  float4 S[C::F];
  auto state_ptr = [&](int h) {
    return reinterpret_cast<float4*>(args.state_pool +
                                     ((size_t)slot * args.h_v + h) * (size_t)(DK * DV));
  };
  // Issue the first head's state loads before the conv so they are in flight
  // while the front end runs.
  {
    const float4* base = state_ptr(hk * G);
#pragma unroll
    for (int m = 0; m < C::F; ++m) S[m] = ld_stream(base + (size_t)(r0 + m * C::RS) * C::CG + cg);
  }

  const IO* __restrict__ xrow = reinterpret_cast<const IO*>(args.x) + (size_t)n * cd;
  IO* __restrict__ win = reinterpret_cast<IO*>(args.conv_pool) + (size_t)slot * 3 * cd;
  for (int e = t; e < 2 * DK; e += C::NT) {
    const int c = e < DK ? hk * DK + e : args.h_k * DK + hk * DK + (e - DK);
    const float y = conv_step<IO>(c, cd, xrow, win, args.conv_weight);
    if (e < DK) s_q[e] = y; else s_k[e - DK] = y;
  }
  __syncthreads();
  if (t < 32) {
    float sq = 0.f, sk = 0.f, qk = 0.f;
    for (int i = t; i < DK; i += 32) {
      sq = fmaf(s_q[i], s_q[i], sq);
      sk = fmaf(s_k[i], s_k[i], sk);
      qk = fmaf(s_q[i], s_k[i], qk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    qk = warp_sum(qk);
    if (t == 0) {
      const float iq = rsqrtf(sq + args.l2_eps) * rsqrtf((float)DK);
      const float ik = rsqrtf(sk + args.l2_eps);
      s_scal[0] = iq;
      s_scal[1] = ik;
      s_scal[2] = qk * iq * ik;  // k^ . q^
    }
  }
  __syncthreads();
  for (int i = t; i < DK; i += C::NT) {
    s_q[i] *= s_scal[0];
    s_k[i] *= s_scal[1];
  }

  for (int gi = 0; gi < G; ++gi) {
    const int h = hk * G + gi;
    float4* base = state_ptr(h);
    if (gi > 0) {
#pragma unroll
      for (int m = 0; m < C::F; ++m) S[m] = ld_stream(base + (size_t)(r0 + m * C::RS) * C::CG + cg);
    }
    for (int j = t; j < DV; j += C::NT)
      s_v[j] = conv_step<IO>(2 * args.h_k * DK + h * DV + j, cd, xrow, win, args.conv_weight);
    const float g = gate_g(ld_io(reinterpret_cast<const IO*>(args.a) + (size_t)n * args.h_v + h),
                           args.A_log[h], args.dt_bias[h]);
    const float alpha = expf(g);
    const float beta = sigmoidf_(ld_io(reinterpret_cast<const IO*>(args.b) + (size_t)n * args.h_v + h));
    // fused gated norm: the gate and weight are fetched now, used after the
    // state write-back
    const size_t oi = ((size_t)n * args.h_v + h) * DV + t;
    float zv = 0.f, wt = 0.f;
    if (fuse && t < DV) {
      zv = ld_io(reinterpret_cast<const IO*>(args.z) + oi);
      wt = args.norm_weight[t];
    }
    __syncthreads();  // s_v written, s_q / s_k normalised

    float u[4] = {0.f, 0.f, 0.f, 0.f}, r[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < C::F; ++m) {
      const int i = r0 + m * C::RS;
      const float ki = s_k[i], qi = s_q[i];
      u[0] = fmaf(S[m].x, ki, u[0]); u[1] = fmaf(S[m].y, ki, u[1]);
      u[2] = fmaf(S[m].z, ki, u[2]); u[3] = fmaf(S[m].w, ki, u[3]);
      r[0] = fmaf(S[m].x, qi, r[0]); r[1] = fmaf(S[m].y, qi, r[1]);
      r[2] = fmaf(S[m].z, qi, r[2]); r[3] = fmaf(S[m].w, qi, r[3]);
    }
    if constexpr (C::CG < 32) {
#pragma unroll
      for (int off = C::CG; off < 32; off <<= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          u[c] += __shfl_xor_sync(0xffffffffu, u[c], off);
          r[c] += __shfl_xor_sync(0xffffffffu, r[c], off);
        }
      }
    }
    const int lane = t & 31, w = t >> 5;
    if (lane < C::CG) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        s_red[0][w][4 * lane + c] = u[c];
        s_red[1][w][4 * lane + c] = r[c];
      }
    }
    __syncthreads();
    float oj = 0.f;   // this thread's output value (j = t < DV)
    if (t < DV) {
      const int j = t;
      float uj = 0.f, rj = 0.f;
#pragma unroll
      for (int ww = 0; ww < C::NW; ++ww) {
        uj += s_red[0][ww][j];
        rj += s_red[1][ww][j];
      }
      const float d = beta * (s_v[j] - alpha * uj);
      s_delta[j] = d;
      oj = fmaf(alpha, rj, d * s_scal[2]);
      if (!fuse) st_io(o + oi, oj);
    }
    if (fuse) {
      // gated RMSNorm over the head's d_v values (the gdn_gated_rmsnorm
      // definition): y = o / sqrt(mean(o^2) + eps) * w * SiLU(z); the per-warp
      // sums of o^2 cross the barrier the state update needs anyway
      const float sq = warp_sum(oj * oj);
      if ((t & 31) == 0 && t < DV) s_nrm[t >> 5] = sq;
    }
    __syncthreads();
    const float4 dl = *reinterpret_cast<const float4*>(&s_delta[4 * cg]);
#pragma unroll
    for (int m = 0; m < C::F; ++m) {
      const int i = r0 + m * C::RS;
      const float ki = s_k[i];
      float4 s;
      s.x = fmaf(alpha, S[m].x, ki * dl.x);
      s.y = fmaf(alpha, S[m].y, ki * dl.y);
      s.z = fmaf(alpha, S[m].z, ki * dl.z);
      s.w = fmaf(alpha, S[m].w, ki * dl.w);
      st_stream(base + (size_t)i * C::CG + cg, s);
    }
    if (fuse && t < DV) {
      float tot = 0.f;
#pragma unroll
      for (int ww = 0; ww < (DV + 31) / 32; ++ww) tot += s_nrm[ww];
      const float inv = rsqrtf(tot * (1.0f / DV) + args.norm_eps);
      st_io(o + oi, oj * inv * wt * silu(zv));
    }
    __syncthreads();  // s_v / s_red / s_delta / s_nrm reused by the next head
  }
}

template <typename IO>
__global__ void __launch_bounds__(256) conv_update_kernel(const GdnConvArgs args) {
  const int n = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= args.conv_dim) return;
  const int slot = args.slot_idx[n];
  IO* y = reinterpret_cast<IO*>(args.y) + (size_t)n * args.conv_dim;
  if (slot < 0 || slot >= args.num_slots) {
    if (slot >= args.num_slots && c == 0) set_status(args.d_status, GDN_DEV_BAD_SLOT);
    st_io(y + c, 0.0f);
    return;
  }
  const IO* xrow = reinterpret_cast<const IO*>(args.x) + (size_t)n * args.conv_dim;
  IO* win = reinterpret_cast<IO*>(args.conv_pool) + (size_t)slot * 3 * args.conv_dim;
  st_io(y + c, conv_step<IO>(c, args.conv_dim, xrow, win, args.conv_weight));
}

template <int DK, int DV, typename IO>
static cudaError_t launch_decode_t(const GdnDecodeArgs& a, cudaStream_t s) {
  using C = DecodeCfg<DK, DV>;
  dim3 grid(a.n, a.h_k);
  decode_step_kernel<DK, DV, IO><<<grid, C::NT, 0, s>>>(a);
  return cudaGetLastError();
}

template <int DK, typename IO>
static cudaError_t launch_decode_dv(const GdnDecodeArgs& a, int d_v, cudaStream_t s) {
  switch (d_v) {
    case 16: return launch_decode_t<DK, 16, IO>(a, s);
    case 32: return launch_decode_t<DK, 32, IO>(a, s);
    case 64: return launch_decode_t<DK, 64, IO>(a, s);
    case 128: return launch_decode_t<DK, 128, IO>(a, s);
  }
  return cudaErrorInvalidValue;
}

template <typename IO>
static cudaError_t launch_decode_io(const GdnDecodeArgs& a, int d_k, int d_v, cudaStream_t s) {
  switch (d_k) {
    case 16: return launch_decode_dv<16, IO>(a, d_v, s);
    case 32: return launch_decode_dv<32, IO>(a, d_v, s);
    case 64: return launch_decode_dv<64, IO>(a, d_v, s);
    case 128: return launch_decode_dv<128, IO>(a, d_v, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gdn

cudaError_t gdn_launch_decode(const GdnDecodeArgs& a, int d_k, int d_v, int io, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  return io == GDN_BF16 ? gdn::launch_decode_io<__nv_bfloat16>(a, d_k, d_v, s)
                        : gdn::launch_decode_io<float>(a, d_k, d_v, s);
}

cudaError_t gdn_launch_conv_update(const GdnConvArgs& a, int io, cudaStream_t s) {
  if (a.n == 0) return cudaSuccess;
  dim3 grid(a.n, (a.conv_dim + 255) / 256);
  if (io == GDN_BF16)
    gdn::conv_update_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
  else
    gdn::conv_update_kernel<float><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}
