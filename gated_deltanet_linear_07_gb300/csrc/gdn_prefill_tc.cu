// gdn_prefill_tc.cu -- tensor-core (tcgen05 / TMEM) chunked prefill for the
// Qwen3.5-4B layer shape: d_k = d_v = 128, chunk 64, bf16 I/O, two value
// heads per key head.
//
// The chunked WY form (oxydllm 0.0.0-alpha.12.2 release notes, New Features,
// "Gated DeltaNet runtime": chunked parallel scan; Performance, "Gated
// DeltaNet fast paths": everything state-independent is batched ahead of the
// cross-chunk loop) runs as two kernels:
//
// prep  one CTA per (chunk, key head), all chunks of all sequences in
//       parallel.  Causal conv + SiLU of the chunk's q, k and both value
//       heads' v (3-token halo from x or from the slot's window), L2 norms,
//       gates and the in-chunk cumulative log-decay gamma; then on the tensor
//       cores  [K;Q] K^T  (one M=128 MMA gives K K^T and Q K^T), the exact
//       inverse T = (I + strict_tril(diag(beta) K K^T * e^{gamma_r-gamma_s}))^-1
//       by blockwise forward substitution in fp32 (finite on fully correlated
//       keys: no matrix powers are formed), and
//         U^T  = V^T  (T diag(beta))^T,      Wk^T = K^T (T diag(beta e^gamma))^T,
//       plus P = tril(Q K^T * e^{gamma_r-gamma_s}).  Results go to the
//       workspace as ready-made shared-memory tile images.
// scan  one CTA per (sequence, value head), sequential over the chunks, with
//       the fp32 state S^T held in registers of the epilogue warps and a bf16
//       copy in shared memory as the MMA operand.  Per chunk (H = S^T):
//         X    = H^T Wk^T                 W^T  = U^T - X
//         O1   = H^T Q^T                  O2   = W^T P^T
//         dH   = (W^T diag(e^{gamma_C - gamma})) K
//         o    = diag(e^gamma) O1^T + O2^T,   H^T <- e^{gamma_C} H^T + dH
//       Chunk inputs stream in with bulk async copies two chunks deep; one
//       thread issues the MMAs; eight epilogue warps own TMEM lanes.
//
// Every mbarrier wait is bounded; on timeout the kernel sets
// GDN_DEV_WAIT_TIMEOUT, skips the dependent work and still frees its TMEM.
#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace tcp {

using namespace gdn::tc;

constexpr int C = 64;     // chunk
constexpr int D = 128;    // d_k = d_v
constexpr uint32_t KQ_BYTES = 128 * 128 * 2;  // [K;Q] tile, K-major, 128 rows
// Record of one (chunk, value head): U^T tile | Wk^T tile | P tile | decay
// factors e^{gamma_r} [64], e^{gamma_C - gamma_r} [64], e^{gamma_C}.
constexpr uint32_t UT_OFF = 0, WK_OFF = 16384, P_OFF = 32768, EXP_OFF = 40960;
constexpr uint32_t VH_REC = 41984;           // per (chunk, value head)
constexpr uint32_t WAIT_LIMIT = 1u << 22;   // suspending try_wait iterations
constexpr uint32_t SPIN_LIMIT = 1u << 26;   // non-blocking test_wait iterations
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float silu_fast(float z) {
  // z * sigmoid(z) with sigmoid(z) = (1 + tanh(z/2)) / 2
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
  return 0.5f * z * (1.0f + t);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Bulk async copies (no tensor map): global -> shared with mbarrier
// completion, shared -> global with bulk-group completion.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// chunk table: chunk_off[b] = sum_{b'<b} ceil(len_b' / C); one CTA.

__global__ void __launch_bounds__(1024) chunk_table_kernel(const GdnPrefillArgs a) {
  __shared__ int32_t s_warp[32];
  if (!a.ws_flag[0]) return;
  const int B = a.num_seqs;
  const int tid = threadIdx.x;
  const int per = (B + 1023) / 1024;
  const int b0 = tid * per;
  int32_t local = 0;
  for (int b = b0; b < b0 + per && b < B; ++b)
    local += (a.cu_seqlens[b + 1] - a.cu_seqlens[b] + C - 1) / C;
  // block-wide exclusive scan of `local`
  const int lane = tid & 31, w = tid >> 5;
  int32_t v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) s_warp[w] = v;
  __syncthreads();
  if (w == 0) {
    int32_t s = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    s_warp[lane] = s;
  }
  __syncthreads();
  int32_t run = v - local + (w > 0 ? s_warp[w - 1] : 0);
  for (int b = b0; b < b0 + per && b < B; ++b) {
    a.chunk_off[b] = run;
    run += (a.cu_seqlens[b + 1] - a.cu_seqlens[b] + C - 1) / C;
  }
  if (tid == 1023) a.chunk_off[B] = run;
}

// ---------------------------------------------------------------------------
// prep: one CTA (512 threads) per (chunk, key head).

struct PrepSmem {
  static constexpr uint32_t KQ = 0;          // 32768  [K;Q] K-major, 128 rows x 128
  static constexpr uint32_t V = 32768;       // 2 x 16384, MN-major (64 rows s x 128 j)
  static constexpr uint32_t A = 65536;       // 2 x fp32 [64][68]; later BU | BW tiles
  static constexpr uint32_t AH = 17408;      // bytes per head of A and of T
  static constexpr uint32_t T = 100352;      // 2 x fp32 [64][68]
  static constexpr uint32_t R = 135168;      // 2 x fp32 [3][16][16]
  static constexpr uint32_t GAM = 141312;    // fp32 [2][64], log2 units
  static constexpr uint32_t BETA = 141824;   // fp32 [2][64]
  static constexpr uint32_t EG = 142336;     // fp32 [2][64], e^{gamma}
  static constexpr uint32_t BAR = 142848;    // 2 mbarriers + tmem address
  static constexpr uint32_t SIZE = BAR + 64;
  static constexpr int AST = 68;             // fp32 row stride of A and T
};

__device__ __forceinline__ int find_seq(const int32_t* __restrict__ off, int B, int32_t gc) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= gc) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(512, 1) prep_kernel(const GdnPrefillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (!a.ws_flag[0]) return;
  const int32_t gc = blockIdx.x;
  const int hk = blockIdx.y;
  const int32_t nch = a.chunk_off[a.num_seqs];
  if (gc >= nch) return;
  const int b = find_seq(a.chunk_off, a.num_seqs, gc);
  const int slot = a.slot_idx[b];
  if (slot < 0 || slot >= a.num_slots) return;  // the scan reports it
  const int c = gc - a.chunk_off[b];
  const int64_t start = a.cu_seqlens[b];
  const int64_t Tb = a.cu_seqlens[b + 1] - start;
  const int64_t t0 = start + (int64_t)c * C;
  const int L = (int)min((int64_t)C, Tb - (int64_t)c * C);
  const bool init = a.has_init ? a.has_init[b] != 0 : false;
  const int cd = a.conv_dim;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + PrepSmem::BAR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + PrepSmem::BAR + 16);
  float* gam = reinterpret_cast<float*>(sm + PrepSmem::GAM);
  float* beta = reinterpret_cast<float*>(sm + PrepSmem::BETA);
  const uint32_t s_base = smem_u32(sm);

  if (warp == 0) {
    tmem_alloc(s_tmem, 256);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }

  // ---- front end: conv + SiLU + L2 norm, one warp per (segment, 8 tokens) ----
  {
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(a.x);
    const __nv_bfloat16* win =
        reinterpret_cast<const __nv_bfloat16*>(a.conv_pool) + (size_t)slot * 3 * cd;
    const int seg = warp >> 3;          // 0: q | k, 1: v of both value heads
    const int r0 = (warp & 7) * 8;
    const int half = lane >> 4, l16 = lane & 15;
    int ch;
    if (seg == 0) ch = half == 0 ? hk * D + 8 * l16 : a.h_k * D + hk * D + 8 * l16;
    else ch = 2 * a.h_k * D + (2 * hk + half) * D + 8 * l16;
    float w[8][4];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 f = *reinterpret_cast<const float4*>(a.conv_weight + 4 * (size_t)(ch + e));
      w[e][0] = f.x; w[e][1] = f.y; w[e][2] = f.z; w[e][3] = f.w;
    }
    // All 11 rows (3-token halo + 8 tokens) are loaded unconditionally from a
    // valid address so the loads issue back to back; masked rows are zeroed
    // afterwards.  Rows before the sequence start come from the slot's window.
    uint4 xr[11];
    bool keep[11];
#pragma unroll
    for (int q = 0; q < 11; ++q) {
      const int rr = r0 - 3 + q;                  // row within the chunk
      const int64_t p = (int64_t)c * C + rr;      // position within the sequence
      const __nv_bfloat16* src = x + (size_t)t0 * cd + ch;  // row 0 of the chunk: always valid
      keep[q] = rr < L && (p >= 0 || init);
      if (rr < L && p >= 0) src = x + (size_t)(t0 + rr) * cd + ch;
      else if (rr < L && init) src = win + (size_t)(3 + p) * cd + ch;
      xr[q] = __ldg(reinterpret_cast<const uint4*>(src));
    }
#pragma unroll
    for (int q = 0; q < 11; ++q)
      if (!keep[q]) xr[q] = make_uint4(0, 0, 0, 0);
    const float qscale = rsqrtf((float)D);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + i;
      float y[8];
      if (r < L) {
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float xv[8];
          bf16x8_to_float(xr[i + k], xv);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = fmaf(w[e][k], xv[e], y[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = silu_fast(y[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = 0.f;
      }
      if (seg == 0) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = (r < L ? rsqrtf(ss + a.l2_eps) : 0.f) * (half == 0 ? qscale : 1.0f);
        const int row = half == 0 ? 64 + r : r;   // rows 0..63 keys, 64..127 queries
        uint4 pk = make_uint4(pack_bf16(y[0] * inv, y[1] * inv), pack_bf16(y[2] * inv, y[3] * inv),
                              pack_bf16(y[4] * inv, y[5] * inv), pack_bf16(y[6] * inv, y[7] * inv));
        st_shared_v4(s_base + PrepSmem::KQ + kmaj_off(128, row, 8 * l16), pk);
      } else {
        uint4 pk = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                              pack_bf16(y[6], y[7]));
        st_shared_v4(s_base + PrepSmem::V + half * 16384 + mnmaj_off(64, 8 * l16, r), pk);
      }
    }
  }
  // ---- gates of the two value heads (warps 14, 15) ----
  unsigned char* vrec0 = a.vh_ws + ((size_t)gc * a.h_v + 2 * hk) * VH_REC;
  float* eg = reinterpret_cast<float*>(sm + PrepSmem::EG);
  if (warp >= 14) {
    const int g = warp - 14;
    const int h = 2 * hk + g;
    const __nv_bfloat16* av = reinterpret_cast<const __nv_bfloat16*>(a.a);
    const __nv_bfloat16* bv = reinterpret_cast<const __nv_bfloat16*>(a.b);
    float gv[2], be[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = 2 * lane + k;
      if (r < L) {
        const size_t idx = (size_t)(t0 + r) * a.h_v + h;
        gv[k] = gate_g(__bfloat162float(av[idx]), a.A_log[h], a.dt_bias[h]);
        be[k] = sigmoidf_(__bfloat162float(bv[idx]));
      } else {
        gv[k] = 0.f;
        be[k] = 0.f;
      }
    }
    const float pair = gv[0] + gv[1];
    float inc = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    const float g0 = (inc - pair + gv[0]) * LOG2E, g1 = inc * LOG2E;  // log2 units
    const float glast = __shfl_sync(0xffffffffu, g1, 31);
    gam[g * 64 + 2 * lane] = g0;
    gam[g * 64 + 2 * lane + 1] = g1;
    beta[g * 64 + 2 * lane] = be[0];
    beta[g * 64 + 2 * lane + 1] = be[1];
    const float e0 = fast_exp2(g0), e1 = fast_exp2(g1);
    eg[g * 64 + 2 * lane] = e0;
    eg[g * 64 + 2 * lane + 1] = e1;
    float* rec = reinterpret_cast<float*>(vrec0 + g * VH_REC + EXP_OFF);
    rec[2 * lane] = e0;
    rec[2 * lane + 1] = e1;
    rec[64 + 2 * lane] = fast_exp2(glast - g0);
    rec[64 + 2 * lane + 1] = fast_exp2(glast - g1);
    if (lane == 0) rec[128] = fast_exp2(glast);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  if (tid == 0) {
    for (int ks = 0; ks < 8; ++ks)
      mma_bf16(tmem, sdesc_kmaj(s_base + PrepSmem::KQ, 128, ks),
               sdesc_kmaj(s_base + PrepSmem::KQ, 128, ks), idesc_bf16(128, 64, false, false),
               ks > 0);
    mma_commit(&bar[0]);
  }
  constexpr int S = PrepSmem::AST;
  // ---- A (rows 0..63 of D1: K K^T) and P (rows 64..127: Q K^T); all warps ----
  {
    const int q = warp & 3, g = (warp >> 2) & 1, sh = warp >> 3;
    const int m = 32 * q + lane;
    const bool ok = mbar_spin(&bar[0], 0, SPIN_LIMIT);
    if (!ok) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
    tc_fence_after();
    float d[32];
    if (ok) tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * sh, d);
    else {
#pragma unroll
      for (int e = 0; e < 32; ++e) d[e] = 0.f;
    }
    const float* gm = gam + g * 64;
    if (m < 64) {
      const int r = m;
      float* A = reinterpret_cast<float*>(sm + PrepSmem::A + g * PrepSmem::AH);
      const float gr = gm[r], br = beta[g * 64 + r];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int s = 32 * sh + e;
        A[r * S + s] = s < r ? br * fast_exp2(gr - gm[s]) * d[e] : 0.f;
      }
    } else {
      const int r = m - 64;
      const float gr = gm[r];
      unsigned char* ptile = vrec0 + g * VH_REC + P_OFF;
#pragma unroll
      for (int ck = 0; ck < 4; ++ck) {
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = 32 * sh + 8 * ck + e;
          pv[e] = s <= r ? fast_exp2(gr - gm[s]) * d[8 * ck + e] : 0.f;
        }
        *reinterpret_cast<uint4*>(ptile + kmaj_off(64, r, 32 * sh + 8 * ck)) =
            make_uint4(pack_bf16(pv[0], pv[1]), pack_bf16(pv[2], pv[3]), pack_bf16(pv[4], pv[5]),
                       pack_bf16(pv[6], pv[7]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // ---- T = (I + A)^-1 per value head: 8 warps per head ----
  {
    const int g = warp >> 3, gt = tid & 255;
    const float* A = reinterpret_cast<const float*>(sm + PrepSmem::A + g * PrepSmem::AH);
    float* T = reinterpret_cast<float*>(sm + PrepSmem::T + g * PrepSmem::AH);
    float* Rt = reinterpret_cast<float*>(sm + PrepSmem::R) + g * 768;
    if (gt < 64) {  // 16x16 diagonal blocks: one column each, forward substitution
      const int kb = gt >> 4, jj = gt & 15, o = kb * 16;
      float tc[16];
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        float acc = 0.f;
#pragma unroll
        for (int ss = 0; ss < rr; ++ss)
          if (ss >= jj) acc = fmaf(A[(o + rr) * S + o + ss], tc[ss], acc);
        tc[rr] = rr < jj ? 0.f : (rr == jj ? 1.f : -acc);
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) T[(o + rr) * S + o + jj] = tc[rr];
    }
    named_bar(1 + g, 256);
    // block rows 1..3: T[bi][bj] = -T[bi][bi] sum_{bk=bj}^{bi-1} A[bi][bk] T[bk][bj];
    // each thread owns a 1x4 strip (row rr, columns 4cg..4cg+3) of one block.
    const int e = gt & 63, rr = e >> 2, cg = e & 3, bj = gt >> 6;
    for (int bi = 1; bi < 4; ++bi) {
      const bool act = bj < bi;
      if (act) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* arow = A + (16 * bi + rr) * S;
        for (int bk = bj; bk < bi; ++bk) {
#pragma unroll
          for (int m2 = 0; m2 < 16; ++m2) {
            const int k = 16 * bk + m2;
            const float av = arow[k];
            const float4 t4 = *reinterpret_cast<const float4*>(T + k * S + 16 * bj + 4 * cg);
            acc.x = fmaf(av, t4.x, acc.x);
            acc.y = fmaf(av, t4.y, acc.y);
            acc.z = fmaf(av, t4.z, acc.z);
            acc.w = fmaf(av, t4.w, acc.w);
          }
        }
        *reinterpret_cast<float4*>(Rt + bj * 256 + rr * 16 + 4 * cg) = acc;
      }
      named_bar(1 + g, 256);
      if (act) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* trow = T + (16 * bi + rr) * S + 16 * bi;
#pragma unroll
        for (int m2 = 0; m2 < 16; ++m2) {
          const float tv = trow[m2];
          const float4 r4 = *reinterpret_cast<const float4*>(Rt + bj * 256 + m2 * 16 + 4 * cg);
          acc.x = fmaf(tv, r4.x, acc.x);
          acc.y = fmaf(tv, r4.y, acc.y);
          acc.z = fmaf(tv, r4.z, acc.z);
          acc.w = fmaf(tv, r4.w, acc.w);
        }
        *reinterpret_cast<float4*>(T + (16 * bi + rr) * S + 16 * bj + 4 * cg) =
            make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
      }
      named_bar(1 + g, 256);
    }
    // B operands of the U / Wk products, (T diag(beta)) and (T diag(beta e^gamma)),
    // written over this head's A (no longer read).
    const uint32_t bu = s_base + PrepSmem::A + g * PrepSmem::AH, bw = bu + 8192;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int chunk = gt + 256 * q;
      const int r = chunk >> 3, s0 = 8 * (chunk & 7);
      float vu[8], vw[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int sc = s0 + k;
        const float t = sc <= r ? T[r * S + sc] : 0.f;
        vu[k] = t * beta[g * 64 + sc];
        vw[k] = vu[k] * eg[g * 64 + sc];
      }
      st_shared_v4(bu + kmaj_off(64, r, s0),
                   make_uint4(pack_bf16(vu[0], vu[1]), pack_bf16(vu[2], vu[3]),
                              pack_bf16(vu[4], vu[5]), pack_bf16(vu[6], vu[7])));
      st_shared_v4(bw + kmaj_off(64, r, s0),
                   make_uint4(pack_bf16(vw[0], vw[1]), pack_bf16(vw[2], vw[3]),
                              pack_bf16(vw[4], vw[5]), pack_bf16(vw[6], vw[7])));
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const uint32_t bu = s_base + PrepSmem::A + g * PrepSmem::AH, bw = bu + 8192;
      for (int ks = 0; ks < 4; ++ks)  // U^T_g -> TMEM columns [64g, 64g+64)
        mma_bf16(tmem + 64 * g, sdesc_mnmaj(s_base + PrepSmem::V + 16384 * g, 64, ks),
                 sdesc_kmaj(bu, 64, ks), idesc_bf16(128, 64, true, false), ks > 0);
      for (int ks = 0; ks < 4; ++ks)  // Wk^T_g -> TMEM columns [128+64g, +64)
        mma_bf16(tmem + 128 + 64 * g, sdesc_mnmaj(s_base + PrepSmem::KQ, 128, ks),
                 sdesc_kmaj(bw, 64, ks), idesc_bf16(128, 64, true, false), ks > 0);
    }
    mma_commit(&bar[1]);
  }
  if (tid == 32) {  // the [K;Q] tile, already in its final image, to the workspace
    bulk_s2g(a.kq_ws + ((size_t)gc * a.h_k + hk) * KQ_BYTES, s_base + PrepSmem::KQ, KQ_BYTES);
  }
  // ---- U^T and Wk^T from TMEM to the workspace ----
  {
    const bool ok = mbar_spin(&bar[1], 0, SPIN_LIMIT);
    if (!ok) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
    tc_fence_after();
    const int q = warp >> 2;             // 0,1: U^T of head q; 2,3: Wk^T of head q-2
    const int m = 32 * (warp & 3) + lane;
    const int g = q & 1;
    unsigned char* dst = vrec0 + g * VH_REC + (q < 2 ? UT_OFF : WK_OFF);
    if (ok) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * q + 32 * h2, v);
#pragma unroll
        for (int ck = 0; ck < 4; ++ck) {
          uint4 pk = make_uint4(pack_bf16(v[8 * ck], v[8 * ck + 1]),
                                pack_bf16(v[8 * ck + 2], v[8 * ck + 3]),
                                pack_bf16(v[8 * ck + 4], v[8 * ck + 5]),
                                pack_bf16(v[8 * ck + 6], v[8 * ck + 7]));
          *reinterpret_cast<uint4*>(dst + kmaj_off(128, m, 32 * h2 + 8 * ck)) = pk;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 32) bulk_wait_read();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// scan: one CTA (576 threads) per (sequence, value head).
//   warp 0: bulk loads of chunk inputs (two buffers)
//   warp 1: MMA issue
//   warps 2..17: epilogue; warp w owns TMEM lanes 32*(w%4).., and group
//               (w-2)/4 takes one quarter of the columns.

struct ScanSmem {
  static constexpr uint32_t BUF = 74752;      // KQ 32768 | UT 16384 | Wk 16384 | P 8192 | exp 1024
  static constexpr uint32_t B_KQ = 0, B_UT = 32768, B_WK = 49152, B_P = 65536, B_EXP = 73728;
  static constexpr uint32_t HT = 2 * BUF;     // 32768, K-major 128 x 128
  static constexpr uint32_t WT = HT + 32768;  // 16384, K-major 128 x 64
  static constexpr uint32_t WTT = WT + 16384; // 16384
  static constexpr uint32_t BAR = WTT + 16384;
  static constexpr uint32_t SIZE = BAR + 256;
};
// TMEM columns
constexpr uint32_t TX = 0, TO1 = 64, TO2 = 128, TDH = 256;
constexpr int SCAN_THREADS = 576;
constexpr uint32_t EPI_THREADS = 512;

__global__ void __launch_bounds__(SCAN_THREADS, 1) scan_kernel(const GdnPrefillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (!a.ws_flag[0]) return;
  const int b = blockIdx.x, h = blockIdx.y, hk = h >> 1;
  const int slot = a.slot_idx[b];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (slot < 0 || slot >= a.num_slots) {
    if (h == 0 && tid == 0 && slot >= a.num_slots) set_status(a.d_status, GDN_DEV_BAD_SLOT);
    return;
  }
  const int64_t start = a.cu_seqlens[b];
  const int64_t Tb = a.cu_seqlens[b + 1] - start;
  const int nch = (int)((Tb + C - 1) / C);
  const int32_t gc0 = a.chunk_off[b];
  const bool init = a.has_init ? a.has_init[b] != 0 : false;
  const uint32_t s_base = smem_u32(sm);

  uint64_t* full = reinterpret_cast<uint64_t*>(sm + ScanSmem::BAR);      // [2]
  uint64_t* empty = full + 2;                                             // [2]
  uint64_t* bar_x = full + 4;
  uint64_t* bar_dh = full + 5;
  uint64_t* bar_o = full + 6;
  uint64_t* wready = full + 7;
  uint64_t* hready = full + 8;
  uint64_t* ofree = full + 9;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(full + 10);
  volatile int* s_abort = reinterpret_cast<volatile int*>(full + 11);

  if (warp == 0) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&empty[0], 1);
    mbar_init(&empty[1], 1);
    mbar_init(bar_x, 1);
    mbar_init(bar_dh, 1);
    mbar_init(bar_o, 1);
    mbar_init(wready, EPI_THREADS);
    mbar_init(hready, EPI_THREADS);
    mbar_init(ofree, EPI_THREADS);
    *s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  float* gstate = a.state_pool + ((size_t)slot * a.h_v + h) * (size_t)(D * D);

  auto fail = [&]() {
    *s_abort = 1;
    set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------- loader ----------------
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        if (c >= 2 && !mbar_wait(&empty[s], ((c >> 1) - 1) & 1, WAIT_LIMIT)) { fail(); break; }
        if (*s_abort) break;
        const uint32_t dst = s_base + s * ScanSmem::BUF;
        mbar_expect_tx(&full[s], ScanSmem::BUF);
        bulk_g2s(dst + ScanSmem::B_KQ, a.kq_ws + ((size_t)(gc0 + c) * a.h_k + hk) * KQ_BYTES,
                 KQ_BYTES, &full[s]);
        bulk_g2s(dst + ScanSmem::B_UT, a.vh_ws + ((size_t)(gc0 + c) * a.h_v + h) * VH_REC,
                 VH_REC, &full[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t ID64 = idesc_bf16(128, 64, false, false);
      constexpr uint32_t ID64_BMN = idesc_bf16(128, 64, false, true);
      constexpr uint32_t ID128_BMN = idesc_bf16(128, 128, false, true);
      const uint64_t d_ht = sdesc_kmaj(s_base + ScanSmem::HT, 128, 0);
      const uint64_t d_wt = sdesc_kmaj(s_base + ScanSmem::WT, 128, 0);
      const uint64_t d_wtt = sdesc_kmaj(s_base + ScanSmem::WTT, 128, 0);
      for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        const uint32_t buf = s_base + s * ScanSmem::BUF;
        const uint64_t d_wk = sdesc_mnmaj(buf + ScanSmem::B_WK, 128, 0);
        const uint64_t d_q = sdesc_kmaj(buf + ScanSmem::B_KQ + 64 * 128, 128, 0);
        const uint64_t d_kmn = sdesc_mnmaj(buf + ScanSmem::B_KQ, 128, 0);
        const uint64_t d_p = sdesc_kmaj(buf + ScanSmem::B_P, 64, 0);
        if (!mbar_spin(&full[s], (c >> 1) & 1, SPIN_LIMIT) ||
            !mbar_spin(hready, c & 1, SPIN_LIMIT)) { fail(); break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // X = H^T Wk^T
          mma_bf16(tmem + TX, sdesc_add(d_ht, (ks >> 2) * 16384 + (ks & 3) * 32),
                   sdesc_add(d_wk, ks * 2048), ID64_BMN, ks > 0);
        mma_commit(bar_x);
        if (c > 0 && !mbar_spin(ofree, (c - 1) & 1, SPIN_LIMIT)) { fail(); break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // O1 = H^T Q^T
          mma_bf16(tmem + TO1, sdesc_add(d_ht, (ks >> 2) * 16384 + (ks & 3) * 32),
                   sdesc_add(d_q, (ks >> 2) * 16384 + (ks & 3) * 32), ID64, ks > 0);
        if (!mbar_spin(wready, c & 1, SPIN_LIMIT)) { fail(); break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // dH = Wt^T K
          mma_bf16(tmem + TDH, sdesc_add(d_wtt, ks * 32), sdesc_add(d_kmn, ks * 2048), ID128_BMN,
                   ks > 0);
        mma_commit(bar_dh);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // O2 = W^T P^T
          mma_bf16(tmem + TO2, sdesc_add(d_wt, ks * 32), sdesc_add(d_p, ks * 32), ID64, ks > 0);
        mma_commit(bar_o);
        mma_commit(&empty[s]);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int grp = (warp - 2) >> 2;            // 0..3
    const uint32_t lbase = (uint32_t)(32 * (warp & 3)) << 16;
    const int j = 32 * (warp & 3) + lane;       // TMEM lane = value index
    float H[32];                                // H^T[j][32*grp + i], fp32
#pragma unroll
    for (int i = 0; i < 32; ++i)
      H[i] = init ? gstate[(size_t)(32 * grp + i) * D + j] : 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4(s_base + ScanSmem::HT + kmaj_off(128, j, 32 * grp + 8 * q),
                   make_uint4(pack_bf16(H[8 * q], H[8 * q + 1]), pack_bf16(H[8 * q + 2], H[8 * q + 3]),
                              pack_bf16(H[8 * q + 4], H[8 * q + 5]),
                              pack_bf16(H[8 * q + 6], H[8 * q + 7])));
    fence_async_smem();
    tc_fence_before();
    mbar_arrive(hready);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o);
    for (int c = 0; c < nch; ++c) {
      if (*s_abort) break;
      const int s = c & 1;
      const uint32_t buf = s_base + s * ScanSmem::BUF;
      const float* ex = reinterpret_cast<const float*>(sm + s * ScanSmem::BUF + ScanSmem::B_EXP);
      const int L = (int)min((int64_t)C, Tb - (int64_t)c * C);
      if (!mbar_spin(&full[s], (c >> 1) & 1, SPIN_LIMIT) || !mbar_spin(bar_x, c & 1, SPIN_LIMIT)) {
        fail();
        break;
      }
      tc_fence_after();
      // W^T = U^T - X and Wt^T = W^T diag(e^{gamma_C - gamma}), r in this group's quarter
      float eg[16];
      const float dec = ex[128];
      {
        float X[16];
        tmem_ld16(tmem + lbase + TX + 16 * grp, X);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int r0 = 16 * grp + 8 * q;
          float u[8];
          bf16x8_to_float(ld_shared_v4(buf + ScanSmem::B_UT + kmaj_off(128, j, r0)), u);
          const float4 e0 = *reinterpret_cast<const float4*>(ex + r0);
          const float4 e1 = *reinterpret_cast<const float4*>(ex + r0 + 4);
          const float4 d0 = *reinterpret_cast<const float4*>(ex + 64 + r0);
          const float4 d1 = *reinterpret_cast<const float4*>(ex + 64 + r0 + 4);
          const float ed[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
          eg[8 * q + 0] = e0.x; eg[8 * q + 1] = e0.y; eg[8 * q + 2] = e0.z; eg[8 * q + 3] = e0.w;
          eg[8 * q + 4] = e1.x; eg[8 * q + 5] = e1.y; eg[8 * q + 6] = e1.z; eg[8 * q + 7] = e1.w;
          float wv[8], wt[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            wv[e] = u[e] - X[8 * q + e];
            wt[e] = wv[e] * ed[e];
          }
          st_shared_v4(s_base + ScanSmem::WT + kmaj_off(128, j, r0),
                       make_uint4(pack_bf16(wv[0], wv[1]), pack_bf16(wv[2], wv[3]),
                                  pack_bf16(wv[4], wv[5]), pack_bf16(wv[6], wv[7])));
          st_shared_v4(s_base + ScanSmem::WTT + kmaj_off(128, j, r0),
                       make_uint4(pack_bf16(wt[0], wt[1]), pack_bf16(wt[2], wt[3]),
                                  pack_bf16(wt[4], wt[5]), pack_bf16(wt[6], wt[7])));
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(wready);
      if (!mbar_spin(bar_dh, c & 1, SPIN_LIMIT)) { fail(); break; }
      tc_fence_after();
      // H^T <- e^{gamma_C} H^T + dH; bf16 copy for the next chunk's MMAs
      {
        float dH[32];
        tmem_ld32(tmem + lbase + TDH + 32 * grp, dH);
#pragma unroll
        for (int e = 0; e < 32; ++e) H[e] = fmaf(dec, H[e], dH[e]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(s_base + ScanSmem::HT + kmaj_off(128, j, 32 * grp + 8 * q),
                     make_uint4(pack_bf16(H[8 * q], H[8 * q + 1]), pack_bf16(H[8 * q + 2], H[8 * q + 3]),
                                pack_bf16(H[8 * q + 4], H[8 * q + 5]),
                                pack_bf16(H[8 * q + 6], H[8 * q + 7])));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(hready);
      if (!mbar_spin(bar_o, c & 1, SPIN_LIMIT)) { fail(); break; }
      tc_fence_after();
      {
        float O1[16], O2[16];
        tmem_ld16(tmem + lbase + TO1 + 16 * grp, O1);
        tmem_ld16(tmem + lbase + TO2 + 16 * grp, O2);
        tc_fence_before();
        mbar_arrive(ofree);
        const int64_t t0 = start + (int64_t)c * C;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = 16 * grp + e;
          if (r < L)
            out[((size_t)(t0 + r) * a.h_v + h) * D + j] = __float2bfloat16_rn(fmaf(eg[e], O1[e], O2[e]));
        }
      }
    }
    if (!*s_abort) {
#pragma unroll
      for (int i = 0; i < 32; ++i) gstate[(size_t)(32 * grp + i) * D + j] = H[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace tcp
}  // namespace gdn

// ---------------------------------------------------------------------------

bool gdn_tc_prefill_supported(int h_k, int h_v, int d_k, int d_v, int chunk, int io) {
  return d_k == 128 && d_v == 128 && chunk == 64 && io == GDN_BF16 && h_v == 2 * h_k;
}

size_t gdn_tc_kq_bytes() { return gdn::tcp::KQ_BYTES; }
size_t gdn_tc_vh_bytes() { return gdn::tcp::VH_REC; }

cudaError_t gdn_launch_prefill_tc(const GdnPrefillArgs& a, cudaStream_t s, gdn_trace* tr) {
  using namespace gdn::tcp;
  cudaError_t e = cudaSuccess;
  if ((e = gdn_trace_mark(tr, 0, true, s)) != cudaSuccess) return e;
  if ((e = gdn_launch_check(a, s, tr)) != cudaSuccess) return e;
  chunk_table_kernel<<<1, 1024, 0, s>>>(a);
  gdn_trace_count(tr, 1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 0, false, s)) != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 1, true, s)) != cudaSuccess) return e;
  if (a.max_chunks > 0) {
    const int smem = (int)PrepSmem::SIZE + 1024;
    e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prep_kernel<<<dim3((unsigned)a.max_chunks, a.h_k), 512, smem, s>>>(a);
    gdn_trace_count(tr, 1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // conv windows are rewritten only after the prep has read them
  if ((e = gdn_launch_window(a, GDN_BF16, s, tr)) != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 1, false, s)) != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 2, true, s)) != cudaSuccess) return e;
  const int smem = (int)ScanSmem::SIZE + 1024;
  e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  scan_kernel<<<dim3(a.num_seqs, a.h_v), SCAN_THREADS, smem, s>>>(a);
  gdn_trace_count(tr, 1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return gdn_trace_mark(tr, 2, false, s);
}
