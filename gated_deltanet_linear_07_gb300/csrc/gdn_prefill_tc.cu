// gdn_prefill_tc.cu -- tensor-core (tcgen05 / TMEM) chunked prefill for the
// Qwen3.5-4B layer shape: d_k = d_v = 128, chunk 64, bf16 I/O, two value
// heads per key head.
//
// The chunked WY form (oxydllm 0.0.0-alpha.12.2 release notes, New Features,
// "Gated DeltaNet runtime": chunked parallel scan; Performance, "Gated
// DeltaNet fast paths": everything state-independent is batched ahead of the
// cross-chunk loop) runs as two kernels:
//
// prep  persistent, one CTA per SM; its 16 warps take one (chunk, key head)
//       item at a time, all chunks of all sequences.  Causal conv + SiLU of
//       the chunk's q, k and both value heads' v (the x rows by TMA, one item
//       ahead; the 3-token halo from x or from the slot's window), gates and
//       the in-chunk cumulative log-decay gamma; then on the tensor cores the
//       [K;Q] Gram matrix (one M=128, N=128 MMA: K K^T, Q K^T and, on its
//       diagonal, the L2 norms, folded into the factors below), the exact
//       inverse T = (I + strict_tril(diag(beta) K K^T * e^{gamma_r-gamma_s}))^-1
//       blockwise (16 x 16 diagonal blocks by fp32 forward substitution, block
//       products on the tensor cores; finite on fully correlated keys: no
//       matrix powers are formed), and
//         U^T  = V^T  (T diag(beta))^T,      Wk^T = K^T (T diag(beta e^gamma))^T,
//       plus P = tril(Q K^T * e^{gamma_r-gamma_s}).  Results go to the
//       workspace as ready-made shared-memory tile images.
// scan  one CTA per (sequence, value head), sequential over the chunks, with
//       the fp32 state S^T held in registers of sixteen chain warps and an
//       fp16 (or bf16) copy in tensor memory as the MMA operand.  Per chunk
//       (H = S^T):
//         X    = H^T Wk^T                 W^T  = U^T - X
//         O1   = H^T Q^T                  O2   = W^T P^T
//         dH   = (W^T diag(e^{gamma_C - gamma})) K
//         o    = diag(e^gamma) O1^T + O2^T,   H^T <- e^{gamma_C} H^T + dH
//       Chunk inputs stream in with bulk async copies two chunks deep; one
//       thread issues the MMAs; sixteen chain warps own TMEM lanes and keep
//       the fp32 state in registers; four output warps write o off the chain.
//
// Every wait is bounded in global time; on timeout the kernel sets
// GDN_DEV_WAIT_TIMEOUT, skips the dependent work and still frees its TMEM.
// Both kernels are instantiated for fp16 (the default) and bf16 MMA operands
// (GDN_BF16_OPERANDS).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "gdn_check.cuh"
#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace tcp {

using namespace gdn::tc;

constexpr int C = 64;     // chunk
constexpr int D = 128;    // d_k = d_v
constexpr uint32_t Q_REC = 2 * 64 * 128 * 2;  // per (chunk, key head): Q tile | K tile, K-major, 64 rows each
constexpr uint32_t K_IN_QREC = 64 * 128 * 2;
// Record of one (chunk, value head), every tile a ready shared-memory image:
//   P    [r][s]  K-major, 64 rows            8 KiB
//   UT   [j][r]  K-major, 128 rows           16 KiB
//   EXP  e^{gamma_r} [64], e^{gamma_C - gamma_r} [64], e^{gamma_C}     1 KiB
//   WK   [r][i]  K-major, 64 rows (two 8 KiB K-blocks)                16 KiB
constexpr uint32_t P_OFF = 0, UT_OFF = 8192, EXP_OFF = 24576, WK_OFF = 25600;
constexpr uint32_t VH_REC = 41984;           // per (chunk, value head)
constexpr uint32_t VH_HEAD = 25600;          // P | UT | EXP, copied in one piece
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float silu_fast(float z) {
  // z * sigmoid(z) with sigmoid(z) = (1 + tanh(z/2)) / 2
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
  return 0.5f * z * (1.0f + t);
}

// Gates on the special-function unit (ex2 / lg2 approximations, a few ulp):
// g = -e^{A_log} softplus(a + dt_bias) with softplus(z) = max(z, 0) +
// ln(1 + e^{-|z|}), and beta = 1 / (1 + e^{-b}).  Their relative error
// (~1e-6) moves the in-chunk decays by far less than the operands' rounding.
__device__ __forceinline__ float lg2_fast(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gate_g_fast(float a, float A_log, float dt_bias) {
  const float z = a + dt_bias;
  const float sp = fmaxf(z, 0.0f) +
                   0.6931471805599453f * lg2_fast(1.0f + fast_exp2(-1.4426950408889634f * fabsf(z)));
  return -fast_exp2(1.4426950408889634f * A_log) * sp;
}
__device__ __forceinline__ float sigmoid_fast(float b) {
  return __fdividef(1.0f, 1.0f + fast_exp2(-1.4426950408889634f * b));
}

// The tensor-core operands of both kernels are fp16 by default (10-bit
// mantissa, range +-65504): the state is multiplied by rounded factors every
// chunk, and fp16 keeps that rounding 8x below bf16's.  GDN_BF16_OPERANDS
// selects bf16 operands instead (the kernels are instantiated for both).
template <bool BF>
struct Op;
template <>
struct Op<false> {   // fp16
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ uint16_t one(float a) {
    __half v = __float2half_rn(a);
    return *reinterpret_cast<uint16_t*>(&v);
  }
  static __device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const __half2* p = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(p[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  static constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
    return idesc_f16(M, N, a_mn, b_mn);
  }
  // warp-level m16n8k16 product, fp32 accumulate
  static __device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                                  const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  static constexpr uint16_t EXP_MASK = 0x7c00u;   // all-ones exponent: Inf / NaN
};
template <>
struct Op<true> {   // bf16
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ uint16_t one(float a) {
    __nv_bfloat16 v = __float2bfloat16_rn(a);
    return *reinterpret_cast<uint16_t*>(&v);
  }
  static __device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
    return idesc_bf16(M, N, a_mn, b_mn);
  }
  static __device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                                  const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  static constexpr uint16_t EXP_MASK = 0x7f80u;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
// Named barrier among `n` threads (whole, converged warps).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}


__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Barrier among the warps working on an item (or one head's four warps) on a
// shared-memory mbarrier that expects one arrival per warp: the warp
// reconverges, lane 0 arrives, everyone waits (bounded) for the phase.  Each
// thread keeps the phase parity it waits for.
struct WarpSet {
  uint32_t bar;     // shared-memory address of the mbarrier
  uint32_t phase;
};
__device__ __forceinline__ bool warpset_sync(WarpSet& w, int lane, uint64_t budget_ns) {
  __syncwarp();
  if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(w.bar) : "memory");
  const bool ok = mbar_wait_addr(w.bar, w.phase, budget_ns);
  w.phase ^= 1u;
  return ok;
}

// Bulk async copies (no tensor map): global -> shared with mbarrier
// completion, shared -> global with bulk-group completion.
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
// All but the four most recently committed copies have read their source.
__device__ __forceinline__ void bulk_wait_read_but4() {
  asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Order this thread's async-proxy global accesses with its generic ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void st_release_gpu(int32_t* p, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Setup, one CTA: validate cu_seqlens (cu[0] = 0, non-decreasing, last =
// total tokens; sets the workspace flag, or the device status bit and no
// flag), then the chunk table chunk_off[b] = sum_{b'<b} ceil(len_b' / C), and
// zero the ready flags.

__global__ void __launch_bounds__(1024) setup_kernel(const GdnPrefillArgs a) {
  __shared__ int32_t s_warp[32];
  __shared__ int s_bad;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int B = a.num_seqs;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = (a.cu_seqlens[0] != 0) || ((int64_t)a.cu_seqlens[B] != a.total_tokens);
  __syncthreads();
  for (int i = tid; i < B; i += 1024)
    if (a.cu_seqlens[i + 1] < a.cu_seqlens[i]) s_bad = 1;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      a.ws_flag[0] = 0;
      set_status(a.d_status, GDN_DEV_BAD_CU_SEQLENS);
    }
    return;
  }
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
  // per-(chunk, key head) ready flags start at zero
  for (int64_t i = tid; i < a.max_chunks * a.h_k; i += 1024) a.chunk_ready[i] = 0;
  if (tid == 0) a.ws_flag[0] = 1;
}

// ---------------------------------------------------------------------------
// prep: persistent CTAs (512 threads), one (chunk, key head) item at a time.

// d (16 x 16, as two 16 x 8 accumulator fragments) += P Q for 16 x 16 fp32
// blocks P (row stride sp, even) and Q (row stride sq) in shared memory: the
// blocks of the chunk inverse, on the tensor cores as m16n8k16 steps with the
// operand type of the call (fp16 carries TF32's 10-bit mantissa at half the
// instructions: one step covers K = 16), fp32 accumulate.
template <bool BF>
__device__ __forceinline__ void mma16x16(float (&d)[2][4], const float* P, int sp, const float* Q,
                                         int sq, int lane) {
  const int gid = lane >> 2, tig = lane & 3;
  auto pk = [](float2 v) { return Op<BF>::pack(v.x, v.y); };
  const uint32_t a[4] = {pk(*reinterpret_cast<const float2*>(P + gid * sp + 2 * tig)),
                         pk(*reinterpret_cast<const float2*>(P + (gid + 8) * sp + 2 * tig)),
                         pk(*reinterpret_cast<const float2*>(P + gid * sp + 2 * tig + 8)),
                         pk(*reinterpret_cast<const float2*>(P + (gid + 8) * sp + 2 * tig + 8))};
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const float* q = Q + 8 * nt + gid;
    const uint32_t b[2] = {Op<BF>::pack(q[(2 * tig) * sq], q[(2 * tig + 1) * sq]),
                           Op<BF>::pack(q[(2 * tig + 8) * sq], q[(2 * tig + 9) * sq])};
    Op<BF>::mma16816(d[nt], a, b);
  }
}
// Store sign * d into a 16 x 16 fp32 block (row stride st).
__device__ __forceinline__ void store16x16(float* Dst, int st, const float (&d)[2][4], float sign,
                                           int lane) {
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    *reinterpret_cast<float2*>(Dst + gid * st + 8 * nt + 2 * tig) =
        make_float2(sign * d[nt][0], sign * d[nt][1]);
    *reinterpret_cast<float2*>(Dst + (gid + 8) * st + 8 * nt + 2 * tig) =
        make_float2(sign * d[nt][2], sign * d[nt][3]);
  }
}

struct PrepSmem {
  static constexpr uint32_t KQ = 0;          // 32768  [K;Q] K-major, 128 rows x 128
  static constexpr uint32_t V = 32768;       // 2 x 16384, MN-major (64 rows s x 128 j)
  static constexpr uint32_t AT = 65536;      // 2 x fp32 [64][68]: A, then T in place; finally
                                             // BU_0 | BU_1 | [BW_0; BW_1] fp16 tiles
  static constexpr uint32_t AH = 17408;      // bytes per head of A / T
  static constexpr uint32_t R = 100352;      // 2 x fp32 [4][16][RST]: inverse products
  static constexpr int RST = 24;             // fp32 row stride of those blocks
  static constexpr uint32_t GAM = R + 2 * 4 * 16 * RST * 4;   // fp32 [2][64], log2 units
  static constexpr uint32_t BETA = GAM + 512;                 // fp32 [2][64]
  static constexpr uint32_t EG = BETA + 512;                  // fp32 [2][64], e^{gamma}
  static constexpr uint32_t DD = EG + 512;                    // fp32 [2][64], e^{gamma_C - gamma}
  // fp32 [128] L2-norm factors (keys 0..63: 1/|k_r|, queries 64..127:
  // d_k^-1/2 / |q_r|), then [2] e^{gamma_C} of the two heads
  static constexpr uint32_t NRM = DD + 512;
  static constexpr uint32_t BAR = NRM + 1024;                 // 2 mbarriers + tmem address
  static constexpr uint32_t SIZE = BAR + 64;
  // The item's x rows, brought in by TMA one item ahead: for each of the four
  // 128-channel segments (q, k, v of value head 2 hk, v of 2 hk + 1) the rows
  // t0 - 3 .. t0 + 63 as a dense [67][128] bf16 box (256-byte rows).
  static constexpr uint32_t XT = (SIZE + 1023) / 1024 * 1024;
  static constexpr uint32_t XT_ROWS = 67;
  static constexpr uint32_t XT_SEG = 17408;                   // 67 x 256 bytes, rounded to 1 KiB
  static constexpr uint32_t XT_BYTES = 4 * XT_ROWS * 256;     // transaction bytes per item
  static constexpr uint32_t SIZE_X0 = XT + 4 * XT_SEG;
  // B operands of the second MMAs: BU_0 | BU_1 | [BW_0; BW_1], fp16 tiles
  // (K-major; the blocks above the diagonal are zeroed once per kernel)
  static constexpr uint32_t BT = SIZE_X0;
  // the CTA's item schedule (SCHED entries of 24 bytes) and 16 warp counts
  static constexpr uint32_t SCH = BT + 32768;
  static constexpr uint32_t SIZE_X = SCH + 512 * 16 + 64;
  static constexpr int AST = 68;             // fp32 row stride of A and T
  static constexpr int THREADS = 256;
};

__device__ __forceinline__ int find_seq(const int32_t* __restrict__ off, int B, int32_t gc) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= gc) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// L2 prefetch of the gates a / b of one work item (rows [t0, t1)), one
// 128-byte line per request, spread over n threads (thread index i).
__device__ __forceinline__ void prefetch_gates(const GdnPrefillArgs& a, int64_t t0, int64_t t1,
                                               int i, int n) {
  const size_t g0 = (size_t)t0 * a.h_v * 2, g1 = (size_t)t1 * a.h_v * 2;  // bytes of a / b rows
  for (size_t o = (g0 & ~(size_t)127) + 128 * (size_t)i; o < g1; o += 128 * (size_t)n) {
    const size_t q = o < g0 ? g0 : o;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const unsigned char*>(a.a) + q) : "memory");
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const unsigned char*>(a.b) + q) : "memory");
  }
}

// One work item of a CTA's schedule: the (chunk, key head) pair and where it
// lives, precomputed into shared memory so that the item loop never waits on
// a lookup in the chunk table.
struct ItemInfo {
  int32_t t0;     // first token
  int32_t gc;     // global chunk
  int32_t slot;   // the sequence's (valid) slot
  uint32_t bits;  // L (bits 0..7) | key head (8..23) | first chunk of its sequence (24) |
                  // initial state (25) | sequence 0 (26)
  __device__ int L() const { return (int)(bits & 0xffu); }
  __device__ int hk() const { return (int)((bits >> 8) & 0xffffu); }
  __device__ bool first() const { return (bits >> 24) & 1u; }
  __device__ bool init() const { return (bits >> 25) & 1u; }
  __device__ bool seq0() const { return (bits >> 26) & 1u; }
};
static_assert(sizeof(ItemInfo) == 16, "schedule entry layout");
constexpr int SCHED = 512;   // schedule entries per refill (one candidate per thread)
// TMA of one item's x rows t0 - 3 .. t0 + 63 of its four channel segments
// into the x tile (rows outside the input read as zero; rows before the
// sequence's start are replaced by the window in the front end).  Issued by
// one thread; completes on `bar` with PrepSmem::XT_BYTES.
__device__ __forceinline__ void issue_x_tile(const GdnPrefillArgs& a, const CUtensorMap* map,
                                             const ItemInfo& p, uint32_t xt, uint64_t* bar) {
  const int y = p.t0 - 3;
  mbar_expect_tx(bar, PrepSmem::XT_BYTES);
  const int hk = p.hk();
  tma_load_2d(xt, map, hk * D, y, bar);                                  // q
  tma_load_2d(xt + PrepSmem::XT_SEG, map, (a.h_k + hk) * D, y, bar);     // k
  tma_load_2d(xt + 2 * PrepSmem::XT_SEG, map, (2 * a.h_k + 2 * hk) * D, y, bar);      // v, 2 hk
  tma_load_2d(xt + 3 * PrepSmem::XT_SEG, map, (2 * a.h_k + 2 * hk + 1) * D, y, bar);  // v, 2 hk + 1
}
// Refill the CTA's schedule with its candidates k0 .. k0 + SCHED - 1 (item
// blockIdx.x + k n of the chunk-major order), keeping the valid ones in order:
// each thread looks one candidate up, a ballot and a block-wide prefix sum
// place it.  Returns the number of entries.  Called by all threads, between
// block barriers.
__device__ int fill_schedule(const GdnPrefillArgs& a, ItemInfo* sched, int32_t* s_cnt, int k0,
                             int n, int n_items, int tid) {
  const int item = (int)blockIdx.x + (k0 + tid) * n;
  ItemInfo e{};
  bool valid = false;
  if (item < n_items) {
    const int32_t gc = item / a.h_k;
    const int b = find_seq(a.chunk_off, a.num_seqs, gc);
    const int slot = a.slot_idx[b];
    valid = slot >= 0 && slot < a.num_slots;
    if (valid) {
      const int32_t c = gc - a.chunk_off[b];
      const int64_t start = a.cu_seqlens[b];
      const int64_t Tb = a.cu_seqlens[b + 1] - start;
      const bool init = a.has_init ? a.has_init[b] != 0 : false;
      e.t0 = (int32_t)(start + (int64_t)c * C);
      e.gc = gc;
      e.slot = slot;
      e.bits = (uint32_t)min((int64_t)C, Tb - (int64_t)c * C) | ((uint32_t)(item % a.h_k) << 8) |
               ((c == 0 ? 1u : 0u) << 24) | ((init ? 1u : 0u) << 25) | ((b == 0 ? 1u : 0u) << 26);
    }
  }
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t vote = __ballot_sync(0xffffffffu, valid);
  if (lane == 0) s_cnt[warp] = __popc(vote);
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < SCHED / 32; ++w) {
    const int cw = s_cnt[w];
    base += w < warp ? cw : 0;
    total += cw;
  }
  if (valid) sched[base + __popc(vote & ((1u << lane) - 1u))] = e;
  __syncthreads();
  return total;
}

// One (chunk, key head) work item, run by the 16 warps of the CTA (thread index
// tid, <= 128 registers each) on ~180 KB of shared memory `sm`, two MMA
// mbarriers (completing once per item; parity ph), the x-tile mbarrier
// (parity xph) and 256 TMEM columns from `tmem`.  The item's x rows are
// already in flight to the x tile (TMA, issued during the previous item);
// once the front end has read them this item issues the next item's tile
// (`next`, or none when next < 0).  One item at a time per SM: the scan
// starts once the first chunk is published, and a 16-warp item takes about
// 60 % of the time of two 8-warp items sharing an SM.  grp synchronises the
// 16 warps, head4 the 4 warps of one value head in the phases that run on
// warps 0..7 only.
constexpr int NW = 16;
constexpr int WPS = NW / 4;             // warps per front-end segment
// The thread that issues the item's record copies (a v warp's: the v warps
// finish the front end first) and, in the next item, waits for them to have
// read shared memory before anyone writes tiles there again.
constexpr int CP_TID = 2 * WPS * 32;
constexpr int TPW = C / WPS;            // tokens per front-end warp
template <bool BF>
__device__ __forceinline__ void prep_item(const GdnPrefillArgs& a, const CUtensorMap* xmap,
                                          const ItemInfo& it, const ItemInfo* next, unsigned char* sm,
                                          int tid, WarpSet& grp, WarpSet& head4, uint64_t* bar,
                                          uint32_t ph, uint64_t* xbar, uint32_t xph, uint32_t tmem,
                                          uint64_t* stg_free) {
  const int32_t gc = it.gc;
  const int hk = it.hk(), slot = it.slot;
  const bool first = it.first();
  const int64_t t0 = it.t0;
  const int L = it.L();
  const bool init = it.init();
  const int cd = a.conv_dim;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int S = PrepSmem::AST;
  float* gam = reinterpret_cast<float*>(sm + PrepSmem::GAM);
  float* beta = reinterpret_cast<float*>(sm + PrepSmem::BETA);
  float* eg = reinterpret_cast<float*>(sm + PrepSmem::EG);
  float* dd = reinterpret_cast<float*>(sm + PrepSmem::DD);
  float* nrm = reinterpret_cast<float*>(sm + PrepSmem::NRM);
  const uint32_t s_base = smem_u32(sm);
  unsigned char* vrec0 = a.vh_ws + ((size_t)gc * a.h_v + 2 * hk) * VH_REC;

  // The gate warps load a and b of the two value heads now and use them after
  // the front end, so that the loads' latency hides behind it.
  const bool gate_warp = warp == 3 * WPS || warp == 3 * WPS + 1;
  uint32_t gab[2] = {0u, 0u};   // (a, b) of tokens 2 lane + k, bf16 pairs
  if (gate_warp) {
    const int h = 2 * hk + warp - 3 * WPS;
    const uint16_t* av = reinterpret_cast<const uint16_t*>(a.a);
    const uint16_t* bv = reinterpret_cast<const uint16_t*>(a.b);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = 2 * lane + k;
      if (r < L) {
        const size_t idx = (size_t)(t0 + r) * a.h_v + h;
        gab[k] = (uint32_t)__ldg(av + idx) | ((uint32_t)__ldg(bv + idx) << 16);
      }
    }
  }
  // ---- front end: conv + SiLU; warp = (segment, TPW tokens), lane = 4 channels ----
  // q and k go into the [K;Q] tile as they are: their L2 norms come from the
  // diagonal of the Gram matrix the first MMA computes, and the factors
  // 1/|q_r|, 1/|k_s| are applied where the products are used.
  if (!mbar_wait(xbar, xph, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
  {
    const __nv_bfloat16* win =
        reinterpret_cast<const __nv_bfloat16*>(a.conv_pool) + (size_t)slot * 3 * cd;
    const int seg = warp / WPS;         // 0: q, 1: k, 2 / 3: v of value head 2 hk / 2 hk + 1
    const int r0 = (warp % WPS) * TPW;
    int ch;
    if (seg == 0) ch = hk * D;
    else if (seg == 1) ch = (a.h_k + hk) * D;
    else ch = 2 * a.h_k * D + (2 * hk + seg - 2) * D;
    ch += 4 * lane;
    // Conv taps as channel pairs, w2[k][p] = (w[ch + 2p][k], w[ch + 2p + 1][k]);
    // the arithmetic below runs on packed fp32 pairs.
    float2 w2[4][2];
#pragma unroll
    for (int p2 = 0; p2 < 2; ++p2) {
      const float4 f0 = __ldg(reinterpret_cast<const float4*>(a.conv_weight + 4 * (size_t)(ch + 2 * p2)));
      const float4 f1 =
          __ldg(reinterpret_cast<const float4*>(a.conv_weight + 4 * (size_t)(ch + 2 * p2 + 1)));
      w2[0][p2] = make_float2(f0.x, f1.x);
      w2[1][p2] = make_float2(f0.y, f1.y);
      w2[2][p2] = make_float2(f0.z, f1.z);
      w2[3][p2] = make_float2(f0.w, f1.w);
    }
    const float2 half2 = make_float2(0.5f, 0.5f);
    auto unpack = [](const uint2& u, float2 (&f)[2]) {
      f[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
      f[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    };
    // This lane's 8 bytes of chunk row r in its tile: q / k rows of the K-major
    // [K;Q] tile (rows 64.. queries, 0.. keys), v the MN-major V tile (token r
    // as the K index); in both the 16-byte piece index is XOR-ed with r % 8.
    const uint32_t tile = seg < 2 ? s_base + PrepSmem::KQ + (lane >> 4) * 16384u +
                                        (seg == 0 ? 64u * 128u : 0u)
                                  : s_base + PrepSmem::V + (seg - 2) * 16384u + (lane >> 4) * 8192u;
    const uint32_t cidx = (uint32_t)(lane & 15) >> 1;
    const uint32_t obase = tile + (uint32_t)r0 * 128u + 8u * (uint32_t)(lane & 1);
    auto out_addr = [&](int i) {   // token r0 + i (r0 is a multiple of 16: r % 8 = i % 8)
      return obase + (uint32_t)i * 128u + ((cidx ^ (uint32_t)(i & 7)) << 4);
    };
    // Rows rr = r0 - 3 .. r0 + TPW - 1 of the chunk: from the x tile (row rr + 3);
    // in a sequence's first chunk the history before its first token comes from
    // the slot's window (or zeros), and rows past the chunk's end are zeros.
    const uint32_t xrow = s_base + PrepSmem::XT + seg * PrepSmem::XT_SEG + 8 * lane;
    const bool interior = !first && L == C;   // every row from the tile
    auto load_row = [&](int rr) -> uint2 {
      if (interior) return ld_shared_v2(xrow + (uint32_t)(rr + 3) * 256u);
      uint2 v = make_uint2(0, 0);
      if (rr < L && (rr >= 0 || !first)) v = ld_shared_v2(xrow + (uint32_t)(rr + 3) * 256u);
      else if (rr < L && init) v = __ldg(reinterpret_cast<const uint2*>(win + (size_t)(3 + rr) * cd + ch));
      return v;
    };
    float2 xf[4][2];
    {
      const uint2 h0 = load_row(r0 - 3), h1 = load_row(r0 - 2), h2 = load_row(r0 - 1);
      unpack(h0, xf[1]);
      unpack(h1, xf[2]);
      unpack(h2, xf[3]);
    }
    uint2 cur[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) cur[i] = load_row(r0 + i);
#pragma unroll
    for (int hh = 0; hh < TPW / 4; ++hh) {
      if (hh == 0) {
        // the previous item's [Q; K] record copies have read the tile this
        // item's q and k go to (signalled by the thread that issued them; its
        // four U / Wk copies, committed after them, may still be reading)
        if (tid == CP_TID) {
          bulk_wait_read_but4();
          mbar_arrive(stg_free);
        }
        if (!mbar_wait(stg_free, xph, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
      }
      const int rb = r0 + 4 * hh;
      uint2 nxt[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) nxt[i] = hh < TPW / 4 - 1 ? load_row(rb + 4 + i) : make_uint2(0, 0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          xf[q][0] = xf[q + 1][0];
          xf[q][1] = xf[q + 1][1];
        }
        unpack(cur[i], xf[3]);
        float2 y[2];   // SiLU(conv) of token rb + i, channel pairs
#pragma unroll
        for (int p2 = 0; p2 < 2; ++p2) {
          float2 z = __fmul2_rn(w2[0][p2], xf[0][p2]);
          z = __ffma2_rn(w2[1][p2], xf[1][p2], z);
          z = __ffma2_rn(w2[2][p2], xf[2][p2], z);
          z = __ffma2_rn(w2[3][p2], xf[3][p2], z);
          // SiLU: z sigmoid(z) = h + h tanh(h), h = z / 2
          const float2 h2 = __fmul2_rn(z, half2);
          float2 t;
          asm("tanh.approx.f32 %0, %1;" : "=f"(t.x) : "f"(h2.x));
          asm("tanh.approx.f32 %0, %1;" : "=f"(t.y) : "f"(h2.y));
          y[p2] = __ffma2_rn(h2, t, h2);
        }
        const uint2 val = interior || rb + i < L
                              ? make_uint2(Op<BF>::pack(y[0].x, y[0].y), Op<BF>::pack(y[1].x, y[1].y))
                              : make_uint2(0, 0);
        st_shared_v2(out_addr(4 * hh + i), val);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
    }
  }
  // The v warps (no norm) finish first: those of value head 2 hk prefetch the
  // next item's gates, two of those of value head 2 hk + 1 compute these.
  if (next && warp >= 2 * WPS && warp < 3 * WPS)
    prefetch_gates(a, next->t0, (int64_t)next->t0 + next->L(), tid - 64 * WPS, 32 * WPS);
  // ---- gates of the two value heads ----
  if (gate_warp) {
    const int g = warp - 3 * WPS;
    const int h = 2 * hk + g;
    float gv[2], be[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = 2 * lane + k;
      if (r < L) {
        gv[k] = gate_g_fast(__uint_as_float(gab[k] << 16), a.A_log[h], a.dt_bias[h]);
        be[k] = sigmoid_fast(__uint_as_float(gab[k] & 0xffff0000u));
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
    const float e0 = fast_exp2(g0), e1 = fast_exp2(g1);
    const float d0 = fast_exp2(glast - g0), d1 = fast_exp2(glast - g1);
    gam[g * 64 + 2 * lane] = g0;
    gam[g * 64 + 2 * lane + 1] = g1;
    beta[g * 64 + 2 * lane] = be[0];
    beta[g * 64 + 2 * lane + 1] = be[1];
    eg[g * 64 + 2 * lane] = e0;
    eg[g * 64 + 2 * lane + 1] = e1;
    dd[g * 64 + 2 * lane] = d0;
    dd[g * 64 + 2 * lane + 1] = d1;
    if (lane == 0) nrm[128 + g] = fast_exp2(glast);
  }
  fence_async_smem();
  tc_fence_before();
  if (!warpset_sync(grp, lane, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
  tc_fence_after();
  // every warp has read the x tile: the next item's rows may land in it
  if (tid == 32 && next) issue_x_tile(a, xmap, *next, s_base + PrepSmem::XT, xbar);
  if (tid == 0) {
    for (int ks = 0; ks < 8; ++ks)  // D1 = [K;Q] [K;Q]^T -> TMEM columns [0, 128)
      mma_ss(tmem, sdesc_kmaj(s_base + PrepSmem::KQ, 128, ks),
             sdesc_kmaj(s_base + PrepSmem::KQ, 128, ks), Op<BF>::idesc(128, 128, false, false),
             ks > 0);
    mma_commit(&bar[0]);
  }
  // ---- L2 norms from the diagonal of D1 (warps 0..3: lane m holds row m) ----
  // n_m = (|x_m|^2 + eps)^-1/2 (x = k_m for m < 64, q_{m-64} scaled by d_k^-1/2
  // otherwise); the records' decay factors take them along: e^{gamma_r} / |q_r|
  // scales the scan's Q-side product, e^{gamma_C - gamma_r} / |k_r| its K side.
  {
    const bool ok = mbar_wait(&bar[0], ph, a.wait_ns);
    if (!ok) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
    tc_fence_after();
    if (warp < 4) {
      const int m = 32 * warp + lane;
      float d[32];
      tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * warp, d);   // column m is d[lane]
      float dg = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) dg = e == lane ? d[e] : dg;
      const float nf = rsqrtf(dg + a.l2_eps) * (m >= 64 ? rsqrtf((float)D) : 1.0f);
      nrm[m] = nf;
      const int r = m & 63;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float* rec = reinterpret_cast<float*>(vrec0 + g * VH_REC + EXP_OFF);
        if (m >= 64) rec[r] = eg[g * 64 + r] * nf;
        else rec[64 + r] = dd[g * 64 + r] * nf;
        if (m == 0) rec[128] = nrm[128 + g];
      }
    }
    // the previous item's U / Wk copies have read their staging (the A/T and
    // B-operand areas this item rewrites from here on)
    if (tid == CP_TID) bulk_wait_read();
    tc_fence_before();
    if (!warpset_sync(grp, lane, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
    tc_fence_after();
  }
  // the B operand tiles start at zero: their blocks above the diagonal stay so
  for (uint32_t o = 16u * tid; o < 32768u; o += 16u * 512u)
    *reinterpret_cast<uint4*>(sm + PrepSmem::BT + o) = make_uint4(0, 0, 0, 0);
  // ---- A (rows 0..63 of D1: K K^T) and P (rows 64..127: Q K^T); warp = (32-column
  //      half, head, lanes) ----
  {
    const int q = warp & 3, g = (warp >> 2) & 1;
    const int m = 32 * q + lane;
    const bool ok = mbar_wait(&bar[0], ph, a.wait_ns);
    if (!ok) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
    tc_fence_after();
    const float* gm = gam + g * 64;
    const int r = m & 63;
    const float gr = gm[r];
    const float nr = nrm[m];   // 1/|k_r| (A rows) or d_k^-1/2 / |q_r| (P rows)
    const float br = beta[g * 64 + r] * nr;
    float* Arow = reinterpret_cast<float*>(sm + PrepSmem::AT + g * PrepSmem::AH) + r * S;
    unsigned char* ptile = vrec0 + g * VH_REC + P_OFF;
    {
      const int hf = warp >> 3;
      float d[32];
      if (ok) {
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * hf, d);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) d[e] = 0.f;
      }
      // the column factors gamma_s and 1/|k_s|, four at a time (float4 broadcasts)
      auto col4 = [&](int c, float (&g4)[4], float (&n4)[4]) {
        const float4 gq = *reinterpret_cast<const float4*>(gm + 32 * hf + c);
        const float4 nq = *reinterpret_cast<const float4*>(nrm + 32 * hf + c);
        g4[0] = gq.x; g4[1] = gq.y; g4[2] = gq.z; g4[3] = gq.w;
        n4[0] = nq.x; n4[1] = nq.y; n4[2] = nq.z; n4[3] = nq.w;
      };
      if (m < 64) {   // A[r][s] = beta_r e^{gamma_r - gamma_s} (k_r . k_s), s < r
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          float av[4], g4[4], n4[4];
          col4(4 * c4, g4, n4);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s2 = 32 * hf + 4 * c4 + e;
            av[e] = s2 < r ? br * fast_exp2(gr - g4[e]) * d[4 * c4 + e] * n4[e] : 0.f;
          }
          *reinterpret_cast<float4*>(Arow + 32 * hf + 4 * c4) = make_float4(av[0], av[1], av[2], av[3]);
        }
      } else {        // P[r][s] = e^{gamma_r - gamma_s} (q_r . k_s), s <= r
#pragma unroll
        for (int ck = 0; ck < 4; ++ck) {
          float pv[8], g4[2][4], n4[2][4];
          col4(8 * ck, g4[0], n4[0]);
          col4(8 * ck + 4, g4[1], n4[1]);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s2 = 32 * hf + 8 * ck + e;
            pv[e] = s2 <= r ? nr * fast_exp2(gr - g4[e >> 2][e & 3]) * d[8 * ck + e] * n4[e >> 2][e & 3]
                            : 0.f;
          }
          *reinterpret_cast<uint4*>(ptile + kmaj_off(64, r, 32 * hf + 8 * ck)) =
              make_uint4(Op<BF>::pack(pv[0], pv[1]), Op<BF>::pack(pv[2], pv[3]), Op<BF>::pack(pv[4], pv[5]),
                         Op<BF>::pack(pv[6], pv[7]));
        }
      }
    }
  }
  tc_fence_before();
  if (!warpset_sync(grp, lane, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
  // ---- T = (I + A)^-1 per value head g on warps 8 g .. 8 g + 7, and the B operands ----
  // With 16 x 16 blocks: D_i = (I + A_ii)^-1 by forward substitution (fp32),
  // then T_10 = -D_1 A_10 D_0 and T_32 = -D_3 A_32 D_2, then the lower-left
  // 32 x 32 block -T_[23][23] R with R = A_[23][01] T_[01][01] (products on the
  // tensor cores as fp16 m16n8k16 steps, fp32 accumulation).  Only products of
  // exact blocks, no matrix powers: finite for fully correlated keys.  T
  // overwrites A block by block; each block's producer also writes its entries
  // of the second MMAs' fp16 B
  // operands BU_g = T diag(beta) and BW_g = T diag(beta e^gamma) (the blocks
  // above the diagonal stay zero from the kernel's start).  The stages of a
  // head meet at its own named barrier.
  {
    const int g = warp >> 3, wl = warp & 7;
    const uint32_t hbar = 1 + g;
    float* AT = reinterpret_cast<float*>(sm + PrepSmem::AT + g * PrepSmem::AH);
    constexpr int RS = PrepSmem::RST;
    float* Rt = reinterpret_cast<float*>(sm + PrepSmem::R) + g * (4 * 16 * RS);
    const float* bt = beta + g * 64;
    const float* et = eg + g * 64;
    const uint32_t bu = s_base + PrepSmem::BT + 8192 * g;   // BU_g: K-major, 64 rows
    const uint32_t bw = s_base + PrepSmem::BT + 16384;      // [BW_0; BW_1]: K-major, 128 rows
    // B entries of -(16 x 16 fragment d) at block (bi, bj)
    auto put_frag = [&](int bi, int bj, const float (&d)[2][4]) {
      const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * bj + 8 * nt + 2 * tig;
        const float b0 = bt[c], b1 = bt[c + 1];
        const float w0 = b0 * et[c] * nrm[c], w1 = b1 * et[c + 1] * nrm[c + 1];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = 16 * bi + gid + 8 * hh;
          const float t0 = -d[nt][2 * hh], t1 = -d[nt][2 * hh + 1];
          st_shared_b32(bu + kmaj_off(64, r, c), Op<BF>::pack(t0 * b0, t1 * b1));
          st_shared_b32(bw + kmaj_off(128, 64 * g + r, c), Op<BF>::pack(t0 * w0, t1 * w1));
        }
      }
    };
    if (wl < 4) {  // D_wl: lane j (< 16) solves column j
      const int o = 16 * wl, j = lane & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float arow[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = *reinterpret_cast<const float4*>(AT + (o + r) * S + o + 4 * q);
          arow[4 * q] = f.x; arow[4 * q + 1] = f.y; arow[4 * q + 2] = f.z; arow[4 * q + 3] = f.w;
        }
        float acc0 = 0.f, acc1 = 0.f;   // two chains: half the dependent latency
#pragma unroll
        for (int s2 = 0; s2 < r; ++s2) {
          if (s2 & 1) acc1 = fmaf(arow[s2], x[s2], acc1);
          else acc0 = fmaf(arow[s2], x[s2], acc0);
        }
        x[r] = r < j ? 0.f : (r == j ? 1.f : -(acc0 + acc1));
      }
      __syncwarp();
      if (lane < 16) {
        const float b0 = bt[o + j], w0 = b0 * et[o + j] * nrm[o + j];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          AT[(o + r) * S + o + j] = x[r];
          st_shared_b16(bu + kmaj_off(64, o + r, o + j), Op<BF>::one(x[r] * b0));
          st_shared_b16(bw + kmaj_off(128, 64 * g + o + r, o + j), Op<BF>::one(x[r] * w0));
        }
      }
    }
    named_bar_sync(hbar, 256);
    if (wl < 2) {  // T_10 (wl 0) and T_32 (wl 1)
      const int i = 1 + 2 * wl;   // block row; column block i - 1
      float* Rw = Rt + wl * 16 * RS;
      float d[2][4] = {};
      mma16x16<BF>(d, AT + 16 * i * S + 16 * (i - 1), S, AT + 16 * (i - 1) * S + 16 * (i - 1), S, lane);
      store16x16(Rw, RS, d, 1.f, lane);
      __syncwarp();
      float e[2][4] = {};
      mma16x16<BF>(e, AT + 16 * i * S + 16 * i, S, Rw, RS, lane);
      store16x16(AT + 16 * i * S + 16 * (i - 1), S, e, -1.f, lane);
      put_frag(i, i - 1, e);
    }
    named_bar_sync(hbar, 256);
    const int bi = 2 + (wl >> 1), bj = wl & 1;   // this warp's block of the lower-left 32 x 32
    if (wl < 4) {  // R_ij = A_i0 T_0j + A_i1 T_1j  (T_01 = 0)
      float d[2][4] = {};
      if (bj == 0) mma16x16<BF>(d, AT + 16 * bi * S, S, AT, S, lane);
      mma16x16<BF>(d, AT + 16 * bi * S + 16, S, AT + 16 * S + 16 * bj, S, lane);
      store16x16(Rt + wl * 16 * RS, RS, d, 1.f, lane);
    }
    named_bar_sync(hbar, 256);
    if (wl < 4) {  // T_ij = -(sum_{k = 2..i} T_ik R_kj): only its B entries are needed
      float d[2][4] = {};
      if (bi == 3) mma16x16<BF>(d, AT + 48 * S + 32, S, Rt + bj * 16 * RS, RS, lane);
      mma16x16<BF>(d, AT + 16 * bi * S + 16 * bi, S, Rt + ((bi - 2) * 2 + bj) * 16 * RS, RS, lane);
      put_frag(bi, bj, d);
    }
  }
  fence_async_smem();
  tc_fence_before();
  if (!warpset_sync(grp, lane, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
  tc_fence_after();
  if (tid == 0) {
#pragma unroll
    for (int g = 0; g < 2; ++g)
      for (int ks = 0; ks < 4; ++ks)  // U^T_g -> TMEM columns [64g, 64g+64)
        mma_ss(tmem + 64 * g, sdesc_mnmaj(s_base + PrepSmem::V + 16384 * g, 64, ks),
               sdesc_kmaj(s_base + PrepSmem::BT + 8192 * g, 64, ks),
               Op<BF>::idesc(128, 64, true, false), ks > 0);
    for (int ks = 0; ks < 4; ++ks)  // [Wk_0; Wk_1] = [BW_0; BW_1] K -> columns [128, 256)
      mma_ss(tmem + 128, sdesc_kmaj(s_base + PrepSmem::BT + 16384, 128, ks),
             sdesc_mnmaj(s_base + PrepSmem::KQ, 128, ks), Op<BF>::idesc(128, 128, false, true),
             ks > 0);
    mma_commit(&bar[1]);
  }
  if (tid == CP_TID) {  // Q rows then K rows of the [K;Q] tile (tile images) to the workspace
    unsigned char* qrec = a.kq_ws + ((size_t)gc * a.h_k + hk) * Q_REC;
    bulk_s2g(qrec, s_base + PrepSmem::KQ + 8192, 8192);
    bulk_s2g(qrec + 8192, s_base + PrepSmem::KQ + 16384 + 8192, 8192);
    bulk_s2g(qrec + K_IN_QREC, s_base + PrepSmem::KQ, 8192);
    bulk_s2g(qrec + K_IN_QREC + 8192, s_base + PrepSmem::KQ + 16384, 8192);
  }
  // ---- U^T and [Wk_0; Wk_1] from TMEM to the workspace ----
  // Staged as the records' tile images in shared memory that nothing reads
  // again this item (the B operands, read by the finished second MMAs, and
  // A/T, dead since the inverse), then written as four 16 KB bulk copies.
  // The next item rewrites those areas only after its front end, the first
  // MMA and the norms, and waits for the copies' reads just before.
  constexpr uint32_t STG_U = PrepSmem::BT;   // U^T_0 | U^T_1
  constexpr uint32_t STG_W = PrepSmem::AT;   // Wk_0 | Wk_1
  {
    const bool ok = mbar_wait(&bar[1], ph, a.wait_ns);
    if (!ok) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
    tc_fence_after();
    const int m = 32 * (warp & 3) + lane;        // TMEM lane of this thread
    // 16 tasks of (lane quarter, 64 columns), one per warp
    if (ok) {
      const int kind = warp >> 2;                // 0,1: U^T_g   2,3: Wk column halves
      const uint32_t col = 64 * kind;
      uint32_t tile;
      int row, R, c0;
      if (kind < 2) {            // U^T_g row j = m
        tile = STG_U + 16384 * kind; row = m; R = 128; c0 = 0;
      } else {                   // Wk of head m/64, row r = m%64, columns i in this half
        tile = STG_W + 16384 * (m >> 6); row = m & 63; R = 64; c0 = 64 * (kind - 2);
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + col + 32 * h2, v);
#pragma unroll
        for (int ck = 0; ck < 4; ++ck) {
          const float* f = &v[8 * ck];
          st_shared_v4(s_base + tile + kmaj_off(R, row, c0 + 32 * h2 + 8 * ck),
                       make_uint4(Op<BF>::pack(f[0], f[1]), Op<BF>::pack(f[2], f[3]), Op<BF>::pack(f[4], f[5]),
                                  Op<BF>::pack(f[6], f[7])));
        }
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  if (!warpset_sync(grp, lane, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
  if (tid == CP_TID) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      bulk_s2g(vrec0 + g * VH_REC + UT_OFF, s_base + STG_U + 16384 * g, 16384);
      bulk_s2g(vrec0 + g * VH_REC + WK_OFF, s_base + STG_W + 16384 * g, 16384);
    }
  }
  // Publish the item when the scan runs beside the prep: every record byte
  // written (bulk stores completed and made visible device-wide, generic
  // stores fenced), then the ready flag with release.  One gpu-scope fence
  // after the group barrier covers every thread's stores (cumulativity), so
  // only thread 0 waits for them.  Without a scan beside the prep nothing is
  // published and the next item starts at once (the kernel waits for the
  // copies' writes before it exits).
  if (a.publish) {
    if (tid == CP_TID) {
      bulk_wait_all();
      fence_proxy_async_global();
    }
    if (!warpset_sync(grp, lane, a.wait_ns)) set_status(a.d_status, GDN_DEV_WAIT_TIMEOUT);
    // (GDN_TEST_WAIT_TIMEOUT: the last chunk of sequence 0, key head 0 stays unpublished)
    const bool withheld = a.withhold_last_chunk && it.seq0() && hk == 0 && gc == a.chunk_off[1] - 1;
    if (tid == 0 && !withheld) {
      __threadfence();
      st_release_gpu(a.chunk_ready + (size_t)gc * a.h_k + hk, 1);
    }
  }
}

// Persistent prep: one CTA per SM, its 16 warps on one (chunk, key head) item
// at a time.  It lets dependent grids (the scan) launch at once.
constexpr uint32_t PREP_SMEM = (PrepSmem::SIZE_X + 1023) / 1024 * 1024;

template <bool BF>
__global__ void __launch_bounds__(512, 1)
    prep_persistent_kernel(const GdnPrefillArgs a, const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint32_t s_tmem;
  // 2 MMA barriers, the 16-warp barrier, 2 head barriers, the x tile, the
  // staging area
  __shared__ __align__(8) uint64_t s_bar[7];
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(&s_tmem, 256);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    mbar_init(&s_bar[2], 16);
    mbar_init(&s_bar[3], 4);
    mbar_init(&s_bar[4], 4);
    mbar_init(&s_bar[5], 1);
    mbar_init(&s_bar[6], 1);   // the staging area is free (once per item)
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The setup kernel's results (flag, chunk table, zeroed counters) are
  // visible after this wait; only then may dependent grids (the scan) start.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!a.ws_flag[0]) {
    if (warp == 0) tmem_dealloc(s_tmem, 256);
    return;
  }
  WarpSet grp16{smem_u32(&s_bar[2]), 0u};
  WarpSet head4{smem_u32(&s_bar[3 + ((tid >> 7) & 1)]), 0u};   // warps 0-3: head 0, 4-7: head 1
  const int32_t nch = a.chunk_off[a.num_seqs];
  const int n_items = nch * a.h_k;
  const int n = (int)gridDim.x;
  uint32_t ph = 0, xph = 0;
  // Static round-robin over the (chunk, key head) items in chunk-major order:
  // in round r, CTA i takes item r n + i, so each round finishes the earliest
  // chunks first.  Items of sequences with an invalid slot are skipped (the
  // scan reports those and waits for nothing).
  // The schedule is refilled every SCHED candidates; the first item of each
  // fill has its x tile issued here, every other one by the item before it.
  ItemInfo* sched = reinterpret_cast<ItemInfo*>(sm + PrepSmem::SCH);
  int32_t* s_cnt = reinterpret_cast<int32_t*>(sm + PrepSmem::SCH + SCHED * sizeof(ItemInfo));
  for (int k0 = 0; (int)blockIdx.x + k0 * n < n_items; k0 += SCHED) {
    __syncthreads();   // every thread is done with the previous fill's entries
    const int cnt = fill_schedule(a, sched, s_cnt, k0, n, n_items, tid);
    if (cnt > 0 && tid == 32) issue_x_tile(a, &xmap, sched[0], smem_u32(sm) + PrepSmem::XT, &s_bar[5]);
    for (int i = 0; i < cnt; ++i) {
      const ItemInfo it = sched[i];
      prep_item<BF>(a, &xmap, it, i + 1 < cnt ? &sched[i + 1] : nullptr, sm, tid, grp16, head4, s_bar,
                ph, &s_bar[5], xph, s_tmem, &s_bar[6]);
      ph ^= 1u;
      xph ^= 1u;
    }
  }
  // the last item's record copies are complete before the CTA exits
  if (tid == CP_TID) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(s_tmem, 256);
}

// ---------------------------------------------------------------------------
// scan: one CTA (704 threads) per (sequence, value head).
//   warp 0: bulk loads of chunk inputs (two buffers)
//   warp 1: MMA issue, four groups per chunk, every A operand in tensor memory
//           (fp16, written by the chain warps), every B operand in shared memory:
//             X  = H^T Wk^T                  (N = 64)
//             O1 = H^T Q^T                   (N = 64, double-buffered)
//             dH = Wt^T K                    (N = 128; Wt = diag(e^{gamma_C-gamma}) W)
//             O2 = W^T P^T                   (N = 64)
//   warps 2..17: the state chain (W and the H update); warp w owns TMEM lanes
//               32*(w%4).., and group (w-2)/4 takes one quarter of the columns.
//   warps 18..21: the output o = e^gamma O1 + O2 of the previous chunk, written
//               while the chain warps work on the next one.

struct ScanSmem {
  // per buffer: P (K-major 64 x 64) | UT | EXP | K (K-major 64 x 128, used MN-major) |
  //             B1 = [Wk; Q] (K-major 128 x 128)
  // B1 is released once X and O1 have read it, the rest once O2 and the chain
  // warps have; the output warps read e^gamma from a copy of their own.
  static constexpr uint32_t BUF = 74752;
  static constexpr uint32_t B_P = 0, B_UT = 8192, B_EXP = 24576, B_K = 25600, B_B1 = 41984;
  static constexpr uint32_t REST = B_B1;      // bytes of P | UT | EXP | K
  static constexpr uint32_t BAR = 2 * BUF;
  static constexpr uint32_t OST = BAR + 256;  // output staging, 2 KiB per output warp
  static constexpr uint32_t EG = OST + 8192;  // e^{gamma} [64] x 2 buffers
  static constexpr uint32_t SIZE = EG + 512;
  // only when checkpointing: a checkpoint's fp32 state [d_k][d_v] (64 KB); the
  // plain call does not reserve it (more of the SM's memory stays L1)
  static constexpr uint32_t CK = SIZE;
  static constexpr uint32_t SIZE_CK = CK + 65536;
  // without checkpoints: the new conv window of this CTA's channels, [3][3 D]
  // bf16, read at the start and written at the end
  static constexpr uint32_t WIN = SIZE;
  static constexpr uint32_t SIZE_WIN = WIN + 3 * 3 * D * 2;
};
// TMEM columns (fp32 accumulators, then the fp16 A operands, two per column):
//   X [64] | O1 x 2 [64] | dH [128] | O2 [64] | H^T [64] | Wt^T [32] | W^T [32]
constexpr uint32_t TX = 0, TO1 = 64, TDH = 192, TO2 = 320, THT = 384, TWT = 448, TW = 480;
constexpr int SCAN_THREADS = 704;
constexpr uint32_t EPI_THREADS = 512;   // the chain warps
constexpr uint32_t OUT_WARPS = 4;

template <bool BF>
__global__ void __launch_bounds__(SCAN_THREADS, 1) scan_kernel(const GdnPrefillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (!a.ws_flag[0]) return;
  const int b = blockIdx.x, h = blockIdx.y, hk = h >> 1;
  const int slot = a.slot_idx[b];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (slot < 0 || slot >= a.num_slots) {
    if (h == 0 && tid == 0) set_status(a.d_status, GDN_DEV_BAD_SLOT);
    return;
  }
  const int64_t start = a.cu_seqlens[b];
  const int64_t Tb = a.cu_seqlens[b + 1] - start;
  const int nch = (int)((Tb + C - 1) / C);
  const int32_t gc0 = a.chunk_off[b];
  const bool init = a.has_init ? a.has_init[b] != 0 : false;
  const uint32_t s_base = smem_u32(sm);
  // Interval checkpoints: the state after chunks ck_every - 1, 2 ck_every - 1,
  // ... (those before the last chunk) goes to slots ck_base, ck_base + 1, ...
  // The chain warps stage it in shared memory before their hready arrival; the
  // MMA issuer, which waits for that arrival anyway, sends it with one bulk
  // copy, walking the checkpoints with a counter (the next checkpoint's chunk):
  // that thread is on the chain and each of its instructions is slow.
  const int32_t ck_every = a.ckpt_every_chunks;
  const int32_t ck_base = ck_every > 0 ? a.ckpt_slot[b] : -1;
  const bool ckpt_on = ck_base >= 0;

  uint64_t* full = reinterpret_cast<uint64_t*>(sm + ScanSmem::BAR);      // [2] P|UT|EXP|K
  uint64_t* empty = full + 2;                                             // [2]
  uint64_t* bar_x = full + 4;
  uint64_t* bar_dh = full + 5;
  uint64_t* wready = full + 6;
  uint64_t* hready = full + 7;
  uint64_t* bar_o = full + 12;                                            // [2]
  uint64_t* ofree = full + 14;                                            // [2]
  uint64_t* full_b1 = full + 16;                                          // [2] [Wk; Q]
  uint64_t* empty_b1 = full + 18;                                         // [2]
  uint64_t* full_eg = full + 20;                                          // [2] e^gamma copy
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(full + 9);
  volatile int* s_abort = reinterpret_cast<volatile int*>(full + 10);

  if (warp == 0) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    // P|UT|EXP|K of a buffer is free once its MMAs are done and every chain
    // warp has read U and the decays; [Wk; Q] once X and O1 are done
    mbar_init(&empty[0], 1 + EPI_THREADS / 32);
    mbar_init(&empty[1], 1 + EPI_THREADS / 32);
    mbar_init(&full_b1[0], 1);
    mbar_init(&full_b1[1], 1);
    mbar_init(&empty_b1[0], 1);
    mbar_init(&empty_b1[1], 1);
    mbar_init(&full_eg[0], 1);
    mbar_init(&full_eg[1], 1);
    mbar_init(bar_x, 1);
    mbar_init(bar_dh, 1);
    mbar_init(&bar_o[0], 1);
    mbar_init(&bar_o[1], 1);
    // the output warps have read O1 and O2 of a TMEM buffer and their e^gamma copy
    mbar_init(&ofree[0], OUT_WARPS);
    mbar_init(&ofree[1], OUT_WARPS);
    // one arrival per chain warp, after its tensor-memory stores are complete
    mbar_init(wready, EPI_THREADS / 32);
    mbar_init(hready, EPI_THREADS / 32);
    *s_abort = 0;
    fence_mbar_init();
  }
  // The sequence's new conv window for this CTA's channels (written at the
  // end): head h's v channels and, from the even head of the pair, key head
  // hk's q and k channels.  Read now, while the first chunk is being prepared.
  const int nch_w = (h & 1) == 0 ? 3 * D : D;
  auto win_channel = [&](int e) {
    return e < D ? 2 * a.h_k * D + h * D + e                                 // v of head h
                 : (e < 2 * D ? hk * D + (e - D) : a.h_k * D + hk * D + (e - 2 * D));   // q, k
  };
  __nv_bfloat16* s_win = reinterpret_cast<__nv_bfloat16*>(sm + ScanSmem::WIN);   // [3][3 D]
  if (a.ckpt_every_chunks == 0) {
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(a.x);
    const __nv_bfloat16* win =
        reinterpret_cast<const __nv_bfloat16*>(a.conv_pool) + (size_t)slot * 3 * a.conv_dim;
    for (int e = tid; e < nch_w; e += SCAN_THREADS) {
      const int c = win_channel(e);
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int64_t tau = Tb - 3 + r;
        s_win[r * 3 * D + e] = tau >= 0 ? x[(size_t)(start + tau) * a.conv_dim + c]
                                        : (init ? win[(size_t)(3 + tau) * a.conv_dim + c]
                                                : __float2bfloat16_rn(0.f));
      }
    }
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
        const uint32_t rel = ((c >> 1) - 1) & 1;   // phase of the release two chunks back
        if (*s_abort) break;
        const uint32_t dst = s_base + s * ScanSmem::BUF;
        if (a.publish) {  // the chunk's records are published by the prep, still running
          const int32_t* fl = a.chunk_ready + (size_t)(gc0 + c) * a.h_k + hk;
          bool late = false;
          if (ld_acquire_gpu(fl) == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(fl) == 0) {
              __nanosleep(64);
              if (globaltimer_ns() - t0 > a.wait_ns) { late = true; break; }
            }
          }
          if (late) { fail(); break; }
          fence_proxy_async_global();
        }
        const unsigned char* vrec = a.vh_ws + ((size_t)(gc0 + c) * a.h_v + h) * VH_REC;
        const unsigned char* qrec = a.kq_ws + ((size_t)(gc0 + c) * a.h_k + hk) * Q_REC;
        if (c >= 2 && !mbar_wait(&empty_b1[s], rel, a.wait_ns)) { fail(); break; }
        mbar_expect_tx(&full_b1[s], ScanSmem::BUF - ScanSmem::REST);
        bulk_g2s(dst + ScanSmem::B_B1, vrec + WK_OFF, 8192, &full_b1[s]);          // Wk K-block 0
        bulk_g2s(dst + ScanSmem::B_B1 + 16384, vrec + WK_OFF + 8192, 8192, &full_b1[s]);  // 1
        bulk_g2s(dst + ScanSmem::B_B1 + 8192, qrec, 8192, &full_b1[s]);            // Q K-block 0
        bulk_g2s(dst + ScanSmem::B_B1 + 24576, qrec + 8192, 8192, &full_b1[s]);    // block 1
        if (c >= 2 && !mbar_wait(&empty[s], rel, a.wait_ns)) { fail(); break; }
        mbar_expect_tx(&full[s], ScanSmem::REST);
        bulk_g2s(dst, vrec, VH_HEAD, &full[s]);                                   // P|UT|EXP
        bulk_g2s(dst + ScanSmem::B_K, qrec + K_IN_QREC, K_IN_QREC, &full[s]);      // K
        if (c >= 2 && !mbar_wait(&ofree[s], rel, a.wait_ns)) { fail(); break; }
        mbar_expect_tx(&full_eg[s], 256);
        bulk_g2s(s_base + ScanSmem::EG + 256 * s, vrec + EXP_OFF, 256, &full_eg[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t ID_XO = Op<BF>::idesc(128, 64, false, false);
      constexpr uint32_t ID_DH = Op<BF>::idesc(128, 128, false, true);
      constexpr uint32_t ID_O2 = Op<BF>::idesc(128, 64, false, false);
      bool ck_reading = false;   // a checkpoint copy may still be reading the staging area
      int ck_next = ck_every - 1;           // chunk after which the next checkpoint falls
      int64_t ck_slot = ck_base;            // and its slot
      for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        const uint32_t buf = s_base + s * ScanSmem::BUF;
        const uint64_t d_b1 = sdesc_kmaj(buf + ScanSmem::B_B1, 128, 0);
        const uint64_t d_k = sdesc_mnmaj(buf + ScanSmem::B_K, 64, 0);
        const uint64_t d_p = sdesc_kmaj(buf + ScanSmem::B_P, 64, 0);
        // Only the two hand-offs of the chain are waited on here, polled without
        // suspending: every barrier operation of this thread is slow while the
        // other warps are busy, so the chain warps certify the rest.  hready (from
        // chain warp 2) also means that [Wk; Q] of this chunk has landed and that
        // O1's buffer has been read; wready that P | U | EXP | K has landed.
        if (!mbar_spin(hready, c & 1, a.wait_ns)) { fail(); break; }
        tc_fence_after();
        if (ckpt_on && c - 1 == ck_next) {   // the checkpoint after chunk c - 1 (c < nch)
          if (ck_slot >= a.num_slots) {
            set_status(a.d_status, GDN_DEV_BAD_SLOT);
          } else {
            bulk_s2g(a.state_pool + ((size_t)ck_slot * a.h_v + h) * (size_t)(D * D),
                     s_base + ScanSmem::CK, 65536);
            ck_reading = true;
          }
          ck_next += ck_every;
          ++ck_slot;
        }
        // A operands advance 16 K elements = 8 columns per step; B operands are
        // 128B-swizzled K-major tiles of 64-element K blocks.
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // X = H^T Wk^T first: it is on the chain
          mma_ts(tmem + TX, tmem + THT + 8 * ks,
                 sdesc_add(d_b1, (ks >> 2) * 16384 + (ks & 3) * 32), ID_XO, ks > 0);
        mma_commit(bar_x);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // O1 = H^T Q^T
          mma_ts(tmem + TO1 + 64 * s, tmem + THT + 8 * ks,
                 sdesc_add(d_b1, 8192 + (ks >> 2) * 16384 + (ks & 3) * 32), ID_XO, ks > 0);
        mma_commit(&empty_b1[s]);
        if (!mbar_spin(wready, c & 1, a.wait_ns)) { fail(); break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // dH = Wt^T K
          mma_ts(tmem + TDH, tmem + TWT + 8 * ks, sdesc_add(d_k, ks * 2048), ID_DH, ks > 0);
        // the chain warps stage the next checkpoint (after this chunk, if there is
        // one) only after bar_dh: the copy has read the staging area by then
        if (ck_reading && c == ck_next && c + 1 < nch) {
          bulk_wait_read();
          ck_reading = false;
        }
        mma_commit(bar_dh);
        // O2 rewrites what the output warps read for the previous chunk
        if (c >= 1 && !mbar_wait(&ofree[s ^ 1], ((c - 1) >> 1) & 1, a.wait_ns)) { fail(); break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // O2 = W^T P^T
          mma_ts(tmem + TO2, tmem + TW + 8 * ks, sdesc_add(d_p, ks * 32), ID_O2, ks > 0);
        mma_commit(&bar_o[s]);
        mma_commit(&empty[s]);
      }
      if (ckpt_on) bulk_wait_all();   // checkpoint copies complete before the CTA exits
    }
  } else if (warp < 2 + (int)(EPI_THREADS / 32)) {
    // ---------------- state chain ----------------
    const int grp = (warp - 2) >> 2;            // 0..3
    const uint32_t lbase = (uint32_t)(32 * (warp & 3)) << 16;
    const int j = 32 * (warp & 3) + lane;       // TMEM lane = value index
    float H[32];                                // H^T[j][32*grp + i], fp32
#pragma unroll
    for (int i = 0; i < 32; ++i)
      H[i] = init ? gstate[(size_t)(32 * grp + i) * D + j] : 0.f;
    // Shared-memory address of this thread's U^T row piece, fixed for the whole scan.
    // In a 128B-swizzled row the consecutive 16-byte pieces q of one 64-column block
    // sit at (first piece) ^ 16 q, so only the first address is kept.
    const uint32_t a_ut0 = ScanSmem::B_UT + kmaj_off(128, j, 16 * grp);   // + buffer base
    // this thread's fp16 A-operand columns: H^T[j][32 grp ..], W^T[j][16 grp ..]
    const uint32_t t_ht = tmem + lbase + THT + 16 * grp;
    const uint32_t t_wt = tmem + lbase + TWT + 8 * grp;
    const uint32_t t_w = tmem + lbase + TW + 8 * grp;
    {
      uint32_t hp[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) hp[e] = Op<BF>::pack(H[2 * e], H[2 * e + 1]);
      tmem_st16(t_ht, hp);
    }
    // warp 2 certifies, through its hready arrivals, what the MMA issuer would
    // otherwise wait for: the next chunk's [Wk; Q] landed, its O1 buffer read
    if (warp == 2 && nch > 0 && !mbar_wait(&full_b1[0], 0, a.wait_ns)) fail();
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(hready);
    for (int c = 0; c < nch; ++c) {
      if (*s_abort) break;
      const int s = c & 1;
      const uint32_t buf = s_base + s * ScanSmem::BUF;
      const uint32_t ex = buf + ScanSmem::B_EXP;   // e^{gamma} [64] | e^{gamma_C - gamma} [64] | e^{gamma_C}
      if (!mbar_wait(&full[s], (c >> 1) & 1, a.wait_ns)) { fail(); break; }
      // U and the decay are loaded while X is computed (the decay factors per row
      // after X: holding them across the wait costs registers).
      const uint4 ut0 = ld_shared_v4(buf + a_ut0), ut1 = ld_shared_v4(buf + (a_ut0 ^ 16u));
      const float dec = ld_shared_f32(ex + 4 * 128);
      if (!mbar_wait(bar_x, c & 1, a.wait_ns)) { fail(); break; }
      tc_fence_after();
      // W^T = U^T - X for r in this group's quarter, and Wt^T = W^T diag(e^{gamma_C - gamma})
      {
        float X[16];
        tmem_ld16(tmem + lbase + TX + 16 * grp, X);
        float edv[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = ld_shared_f4(ex + 4 * (64 + 16 * grp + 4 * q));
          edv[4 * q] = f.x; edv[4 * q + 1] = f.y; edv[4 * q + 2] = f.z; edv[4 * q + 3] = f.w;
        }
        uint32_t wp[8], wtp[8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float u[8];
          Op<BF>::unpack8(q == 0 ? ut0 : ut1, u);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float w0 = u[e] - X[8 * q + e], w1 = u[e + 1] - X[8 * q + e + 1];
            wp[4 * q + e / 2] = Op<BF>::pack(w0, w1);
            wtp[4 * q + e / 2] = Op<BF>::pack(w0 * edv[8 * q + e], w1 * edv[8 * q + e + 1]);
          }
        }
        tmem_st8(t_wt, wtp);
        tmem_st8(t_w, wp);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(wready);
          mbar_arrive(&empty[s]);   // U and the decays of buffer s are read
        }
      }
      if (warp == 2 && c + 1 < nch) {   // idle until dH: certify the next chunk's inputs
        const int s1 = (c + 1) & 1;
        if (!mbar_wait(&full_b1[s1], ((c + 1) >> 1) & 1, a.wait_ns) ||
            (c + 1 >= 2 && !mbar_wait(&ofree[s1], (((c + 1) >> 1) - 1) & 1, a.wait_ns))) {
          fail();
          break;
        }
      }

      if (!mbar_wait(bar_dh, c & 1, a.wait_ns)) { fail(); break; }
      tc_fence_after();
      // H^T <- e^{gamma_C} H^T + dH; fp16 copy for the next chunk's MMAs
      {
        float dH[32];
        tmem_ld32(tmem + lbase + TDH + 32 * grp, dH);
        const float2 dd = make_float2(dec, dec);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 r2 = __ffma2_rn(dd, make_float2(H[2 * e], H[2 * e + 1]),
                                       make_float2(dH[2 * e], dH[2 * e + 1]));
          H[2 * e] = r2.x;
          H[2 * e + 1] = r2.y;
        }
      }
      {
        uint32_t hp[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) hp[e] = Op<BF>::pack(H[2 * e], H[2 * e + 1]);
        tmem_st16(t_ht, hp);
      }
      if (ckpt_on && (c + 1) % ck_every == 0 && c + 1 < nch) {   // stage it, [i][j] as in the pool
        float* ck = reinterpret_cast<float*>(sm + ScanSmem::CK);
#pragma unroll
        for (int i = 0; i < 32; ++i) ck[(32 * grp + i) * D + j] = H[i];
        fence_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(hready);
    }
    if (!*s_abort) {
#pragma unroll
      for (int i = 0; i < 32; ++i) gstate[(size_t)(32 * grp + i) * D + j] = H[i];
    }
  } else {
    // ---------------- output ----------------
    // o[t][h][j] = e^{gamma_r} O1[j][r] + O2[j][r] for the chunk's tokens r.  This
    // warp holds the values j = 32 (w % 4) + lane; it stages 16 tokens at a time in
    // its own 2 KiB (two 1 KiB halves, alternating) and writes them as 16-byte
    // pieces, 8 values of one token each.
    const uint32_t lbase = (uint32_t)(32 * (warp & 3)) << 16;
    const int ow = warp - 2 - (int)(EPI_THREADS / 32);   // 0..3
    const size_t o_row = (size_t)a.h_v * D;
    // this lane's piece: token e = lane/4 (+8), values 8 (lane % 4) .. of the warp's 32
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(a.o) +
                        ((size_t)(start + (lane >> 2)) * a.h_v + h) * D + 32 * (warp & 3) +
                        8 * (lane & 3);
    for (int c = 0; c < nch; ++c) {
      if (*s_abort) break;
      const int s = c & 1;
      const uint32_t ex = s_base + ScanSmem::EG + 256 * s;   // e^{gamma} [64]
      const int L = (int)min((int64_t)C, Tb - (int64_t)c * C);
      if (!mbar_wait(&full_eg[s], (c >> 1) & 1, a.wait_ns) ||
          !mbar_wait(&bar_o[s], (c >> 1) & 1, a.wait_ns)) { fail(); break; }
      tc_fence_after();
#pragma unroll 1
      for (int g = 0; g < C / 16; ++g) {
        float O1[16], O2[16];
        tmem_ld16x2(tmem + lbase + TO1 + 64 * s + 16 * g, O1, tmem + lbase + TO2 + 16 * g, O2);
        float eg[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = ld_shared_f4(ex + 4 * (16 * g + 4 * q));
          eg[4 * q] = f.x; eg[4 * q + 1] = f.y; eg[4 * q + 2] = f.z; eg[4 * q + 3] = f.w;
        }
        __nv_bfloat16* ost =
            reinterpret_cast<__nv_bfloat16*>(sm + ScanSmem::OST + ow * 2048 + (g & 1) * 1024);
#pragma unroll
        for (int e = 0; e < 16; ++e) ost[e * 32 + lane] = __float2bfloat16_rn(fmaf(eg[e], O1[e], O2[e]));
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int e = (lane >> 2) + 8 * q;
          if (16 * g + e < L)
            *reinterpret_cast<uint4*>(ob + (size_t)(16 * g + 8 * q) * o_row) =
                *reinterpret_cast<const uint4*>(ost + e * 32 + 8 * (lane & 3));
        }
        __syncwarp();   // this half is rewritten two groups later
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofree[s]);
      ob += (size_t)C * o_row;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
  // The new conv window read at the start goes out.  The one reader of the old
  // rows, chunk 0's prep item of key head hk, published before this CTA
  // consumed chunk 0.  With checkpoints the window kernel writes every window
  // (it also writes the checkpoints').
  if (a.ckpt_every_chunks == 0 && !*s_abort) {
    __nv_bfloat16* win =
        reinterpret_cast<__nv_bfloat16*>(a.conv_pool) + (size_t)slot * 3 * a.conv_dim;
    for (int e = tid; e < nch_w; e += SCAN_THREADS) {
      const int c = win_channel(e);
#pragma unroll
      for (int r = 0; r < 3; ++r) win[(size_t)r * a.conv_dim + c] = s_win[r * 3 * D + e];
    }
  }
  // Launched as a dependent of the prep, finish only after it (a no-op otherwise).
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace tcp
}  // namespace gdn

// ---------------------------------------------------------------------------

bool gdn_tc_prefill_supported(int h_k, int h_v, int d_k, int d_v, int chunk, int io) {
  return d_k == 128 && d_v == 128 && chunk == 64 && io == GDN_BF16 && h_v == 2 * h_k;
}

size_t gdn_tc_kq_bytes() { return gdn::tcp::Q_REC; }
size_t gdn_tc_vh_bytes() { return gdn::tcp::VH_REC; }

namespace gdn {
namespace tcp {

// GDN_CHECK_FINITE scan of the chunk records (gdn_check.cuh): block (gc, y)
// takes chunk gc's [Q; K] record of key head y (y < h_k, the front end's
// output) or the record of value head y - h_k (the chunk stage's output: P,
// U^T, the 129 decay factors, Wk).
template <bool BF>
__global__ void __launch_bounds__(256) check_records_kernel(const GdnPrefillArgs a) {
  if (!a.ws_flag[0]) return;
  const int gc = blockIdx.x, y = blockIdx.y;
  const int B = a.num_seqs;
  if (gc >= a.chunk_off[B]) return;
  int lo = 0, hi = B - 1;   // the largest b with chunk_off[b] <= gc
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.chunk_off[mid] <= gc) lo = mid; else hi = mid - 1;
  }
  const int slot = a.slot_idx[lo];
  if (slot < 0 || slot >= a.num_slots) return;
  auto f16_bad = [](const unsigned char* p, int n, int tid, int nt) {   // operand Inf / NaN
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
    bool bad = false;
    for (int e = tid; e < n; e += nt) bad |= (q[e] & Op<BF>::EXP_MASK) == Op<BF>::EXP_MASK;
    return bad;
  };
  const int tid = threadIdx.x, nt = blockDim.x;
  bool bad;
  if (y < a.h_k) {
    bad = f16_bad(a.kq_ws + ((size_t)gc * a.h_k + y) * Q_REC, Q_REC / 2, tid, nt);
  } else {
    const unsigned char* rec = a.vh_ws + ((size_t)gc * a.h_v + (y - a.h_k)) * VH_REC;
    bad = f16_bad(rec + P_OFF, (UT_OFF - P_OFF) / 2, tid, nt) ||
          f16_bad(rec + UT_OFF, (EXP_OFF - UT_OFF) / 2, tid, nt) ||
          f16_bad(rec + WK_OFF, (VH_REC - WK_OFF) / 2, tid, nt);
    const uint32_t* ex = reinterpret_cast<const uint32_t*>(rec + EXP_OFF);
    for (int e = tid; e < 2 * C + 1; e += nt) bad |= (ex[e] & 0x7f800000u) == 0x7f800000u;
  }
  if (__syncthreads_or(bad) && tid == 0)
    set_status(a.d_status, y < a.h_k ? GDN_DEV_NONFINITE_FRONTEND : GDN_DEV_NONFINITE_CHUNK);
}

}  // namespace tcp
}  // namespace gdn

cudaError_t gdn_check_tc_records(const GdnPrefillArgs& a, cudaStream_t s) {
  if (a.total_tokens == 0) return cudaSuccess;
  const dim3 grid((unsigned)a.max_chunks, a.h_k + a.h_v);
  if (a.bf16_ops)
    gdn::tcp::check_records_kernel<true><<<grid, 256, 0, s>>>(a);
  else
    gdn::tcp::check_records_kernel<false><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on the driver library).
void* gdn_tensor_map_encoder() {
  static void* const fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<void*>(nullptr);
    return p;
  }();
  return fn;
}

// Tensor map of x [total_tokens][conv_dim] bf16 for the prep's tiles: boxes of
// 128 channels x 67 rows, dense (no swizzle), zero fill outside the input.
static cudaError_t make_x_map(const GdnPrefillArgs& a, CUtensorMap* map) {
  const auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(gdn_tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)a.conv_dim,
                              (cuuint64_t)(a.total_tokens > 0 ? a.total_tokens : 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)a.conv_dim * 2};
  const cuuint32_t box[2] = {128, gdn::tcp::PrepSmem::XT_ROWS};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t gdn_launch_prefill_tc(const GdnPrefillArgs& a_in, cudaStream_t s, gdn_trace* tr) {
  using namespace gdn::tcp;
  cudaError_t e = cudaSuccess;
  GdnPrefillArgs a = a_in;
  CUtensorMap xmap;
  if ((e = make_x_map(a, &xmap)) != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  // With few (sequence, head) chains the scan leaves most SMs idle: run the
  // prep on the other SMs at the same time and let the scan consume chunks
  // as they are published.  Otherwise the prep gets every SM first.
  const int64_t n_scan = (int64_t)a.num_seqs * a.h_v;
  const bool overlap = n_scan <= n_sm / 2;
  // (GDN_TEST_WAIT_TIMEOUT withholds a published flag: only where flags exist)
  if (!overlap) a.withhold_last_chunk = 0;
  a.publish = overlap ? 1 : 0;
  const int workers = overlap ? n_sm - (int)n_scan : n_sm;
  const int psmem = (int)PREP_SMEM + 1024;
  const int ssmem =
      (int)(a.ckpt_every_chunks > 0 ? ScanSmem::SIZE_CK : ScanSmem::SIZE_WIN) + 1024;
  // the fp16 or the bf16 instantiation (GDN_BF16_OPERANDS)
  auto prep_fn = a.bf16_ops ? prep_persistent_kernel<true> : prep_persistent_kernel<false>;
  auto scan_fn = a.bf16_ops ? scan_kernel<true> : scan_kernel<false>;
  if ((e = cudaFuncSetAttribute(prep_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(scan_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ssmem)) !=
      cudaSuccess)
    return e;

  if ((e = gdn_trace_mark(tr, 0, true, s)) != cudaSuccess) return e;
  setup_kernel<<<1, 1024, 0, s>>>(a);
  gdn_trace_count(tr, 1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = gdn_trace_mark(tr, 0, false, s)) != cudaSuccess) return e;
  // the prep is a programmatic dependent of the setup (it waits for it on
  // the device) and the scan, when overlapped, of the prep
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3(workers);
  pcfg.blockDim = dim3(512);
  pcfg.dynamicSmemBytes = psmem;
  pcfg.stream = s;
  pcfg.attrs = attr;
  pcfg.numAttrs = tr ? 0 : 1;   // a stage event between the two ends the overlap anyway

  if (!overlap) {
    if ((e = gdn_trace_mark(tr, 1, true, s)) != cudaSuccess) return e;
    if ((e = cudaLaunchKernelEx(&pcfg, prep_fn, a, xmap)) != cudaSuccess) return e;
    gdn_trace_count(tr, 1);
    if ((e = gdn_trace_mark(tr, 1, false, s)) != cudaSuccess) return e;
    if ((e = gdn_trace_mark(tr, 2, true, s)) != cudaSuccess) return e;
    scan_fn<<<dim3(a.num_seqs, a.h_v), SCAN_THREADS, ssmem, s>>>(a);
    gdn_trace_count(tr, 1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else {
    // stage 2 covers prep and scan together: no event may sit between them
    if ((e = gdn_trace_mark(tr, 2, true, s)) != cudaSuccess) return e;
    if ((e = cudaLaunchKernelEx(&pcfg, prep_fn, a, xmap)) != cudaSuccess) return e;
    gdn_trace_count(tr, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_seqs, a.h_v);
    cfg.blockDim = dim3(SCAN_THREADS);
    cfg.dynamicSmemBytes = ssmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, scan_fn, a)) != cudaSuccess) return e;
    gdn_trace_count(tr, 1);
  }
  // With checkpoints the window kernel writes the sequences' windows and the
  // checkpoints' after the scan; otherwise the scan wrote them itself.
  if (a.ckpt_every_chunks > 0 && (e = gdn_launch_window(a, GDN_BF16, s, tr)) != cudaSuccess)
    return e;
  return gdn_trace_mark(tr, 2, false, s);
}
