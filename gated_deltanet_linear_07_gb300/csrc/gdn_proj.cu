// gdn_proj.cu -- the decay and beta input projections of the layer as one
// matmul over the whole token batch (oxydllm 0.0.0-alpha.12.2 release notes,
// Performance, "Gated DeltaNet fast paths": the small beta/decay projections
// fuse into one matmul).  With W = [W_a; W_b] (2 h_v rows of d_model):
//   [a | b][t] = hidden[t] W^T,   a, b  [n][h_v] bf16
// the gate inputs that gdn_prefill and gdn_decode_step read.
//
// Tensor cores: a CTA owns 128 tokens (the MMA's M) and all N = 2 h_v
// outputs, and streams K = d_model in 64-element blocks by TMA (128-byte
// swizzled rows) through as many stages as shared memory holds, so that all
// of its blocks are in flight at once at the 4B shape.  The op is HBM-bound on
// reading `hidden`, so a tile's K blocks are split over a cluster of up to four
// CTAs (four times the bytes in flight); the partial sums are reduce-scattered
// through distributed shared memory: each rank pushes the 16-column groups
// that another rank owns into that rank's shared memory, then sums and writes
// the groups it owns, rounded once to bf16.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace proj {

using namespace gdn::tc;

constexpr int TM = 128;          // tokens per tile (the MMA's M, one TMEM lane each)
constexpr int KB = 64;           // K elements per stage: one 128-byte swizzled row
constexpr int MAX_STAGES = 8;
constexpr uint32_t SMEM_BYTES = 220 * 1024;   // stages + pushed partials
constexpr int THREADS = 128;
constexpr int MAX_SPLIT = 4;     // K split over a cluster of at most this many CTAs
constexpr uint32_t A_BYTES = TM * KB * 2;
// A pushed 16-column partial: one 64-byte row per token, padded to 80 bytes
// (conflict-free 16-byte accesses by consecutive tokens).
constexpr uint32_t SLOT_ROW = 80;

struct ProjArgs {
  void* a;
  void* b;
  int32_t* d_status;
  int64_t n;
  int32_t h_v;
  int32_t nkb;      // K blocks of 64
  int32_t split;    // cluster size along y
  int32_t stages;   // pipeline depth, <= MAX_STAGES
  uint32_t slots;   // byte offset of the pushed-partials area (after the stages)
  uint64_t wait_ns;
};

__device__ __forceinline__ float4 ld_shared_f4v(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  return remote;
}
// 16 fp32 to a shared::cluster address (another CTA's shared memory).
__device__ __forceinline__ void st_cluster_16(uint32_t remote, const float (&v)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote + 16u * k),
                 "f"(v[4 * k]), "f"(v[4 * k + 1]), "f"(v[4 * k + 2]), "f"(v[4 * k + 3])
                 : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's earlier writes to the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}
// Bounded wait on a local mbarrier whose arrivals come from other CTAs of
// the cluster (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t budget_ns) {
  const uint32_t addr = smem_u32(bar);
  auto test = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (test()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!test())
    if (globaltimer_ns() - t0 > budget_ns) return false;
  return true;
}

__global__ void __launch_bounds__(THREADS)
    gate_projection_kernel(const ProjArgs p, const __grid_constant__ CUtensorMap hmap,
                           const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // full, empty per stage, the accumulator done, the pushed partials landed
  __shared__ __align__(8) uint64_t bars[2 * MAX_STAGES + 2];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const uint32_t rank = cluster_rank();
  const int N = 2 * p.h_v;
  const uint32_t stage_bytes = A_BYTES + (uint32_t)N * KB * 2;
  const uint32_t ncols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;
  const int STAGES = p.stages;
  uint64_t* full = bars;
  uint64_t* empty = bars + MAX_STAGES;
  uint64_t* done = bars + 2 * MAX_STAGES;
  uint64_t* landed = bars + 2 * MAX_STAGES + 1;
  const uint32_t base = smem_u32(sm);
  // this CTA's K blocks: rank, rank + split, rank + 2 split, ...
  const int my = (p.nkb - (int)rank + p.split - 1) / p.split;
  bool ok = true;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    // every thread of every other rank pushes once (unused without a split)
    mbar_init(landed, p.split > 1 ? (uint32_t)(p.split - 1) * THREADS : 1u);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, ncols);
    tmem_relinquish();
  }
  // the barriers are initialised before any other rank arrives on `landed`
  // (this arrival pairs with the wait before the pushes)
  if (p.split > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (tid == 0) {
    // ---- TMA producer: the tile's hidden rows and the weight rows, per K block ----
    for (int i = 0; i < my; ++i) {
      const int s = i % STAGES;
      if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t st = base + (uint32_t)s * stage_bytes;
      const int kx = ((int)rank + i * p.split) * KB;
      mbar_expect_tx(&full[s], stage_bytes);
      tma_load_2d(st, &hmap, kx, tile * TM, &full[s]);
      tma_load_2d(st + A_BYTES, &wmap, kx, 0, &full[s]);
    }
  } else if (tid == 32) {
    // ---- MMA issuer: D[t][r] += hidden[t][k..] W[r][k..], four K=16 steps per block ----
    const uint32_t idesc = idesc_bf16(TM, N, false, false);
    for (int i = 0; i < my; ++i) {
      const int s = i % STAGES;
      if (!mbar_wait(&full[s], (i / STAGES) & 1, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t st = base + (uint32_t)s * stage_bytes;
#pragma unroll
      for (int ks = 0; ks < KB / 16; ++ks)
        mma_ss(tmem, sdesc_kmaj(st, TM, ks), sdesc_kmaj(st + A_BYTES, N, ks), idesc,
               (i > 0 || ks > 0) ? 1u : 0u);
      mma_commit(&empty[s]);
    }
    // arrives once everything issued above has completed (also after a failed wait)
    mma_commit(done);
  }
  __syncwarp();
  const bool got = mbar_wait(done, 0, p.wait_ns);
  tc_fence_after();
  if (!ok || !got) set_status(p.d_status, GDN_DEV_WAIT_TIMEOUT);

  // ---- reduce-scatter of the partial sums over the cluster ----
  // TMEM lane = token within the tile; warp w reads lanes 32 w .. 32 w + 31.
  // 16-column group g belongs to rank g % split.  Its owner's area holds one
  // slot per (other source rank, owned group); each source pushes its
  // partials there and then arrives on the owner's `landed` barrier.
  const uint32_t lrow = (uint32_t)(32 * warp) << 16;
  const int tl = 32 * warp + lane;
  const int G = N / 16;
  const int gpr = (G + p.split - 1) / p.split;   // groups owned per rank, at most
  auto slot = [&](int src, int owner, int lg) {   // in the owner's shared memory
    const int si = src < owner ? src : src - 1;
    return base + p.slots + ((uint32_t)(si * gpr + lg) * TM + (uint32_t)tl) * SLOT_ROW;
  };
  if (p.split > 1) {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    for (int g = 0; g < G; ++g) {
      const int owner = g % p.split;
      if (owner == (int)rank) continue;
      float v[16];
      tmem_ld16(tmem + lrow + 16u * (uint32_t)g, v);
      st_cluster_16(map_to_rank(slot((int)rank, owner, g / p.split), (uint32_t)owner), v);
    }
    for (int r = 0; r < p.split; ++r)
      if (r != (int)rank) mbar_arrive_remote(map_to_rank(smem_u32(landed), (uint32_t)r));
    if (!mbar_wait_cluster(landed, 0, p.wait_ns)) set_status(p.d_status, GDN_DEV_WAIT_TIMEOUT);
  }
  const int64_t t = (int64_t)tile * TM + tl;
  for (int g = (int)rank; g < G; g += p.split) {
    float v[16];
    tmem_ld16(tmem + lrow + 16u * (uint32_t)g, v);
    for (int src = 0; src < p.split; ++src) {
      if (src == (int)rank) continue;
      const uint32_t sa = slot(src, (int)rank, g / p.split);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 f = ld_shared_f4v(sa + 16u * k);
        v[4 * k] += f.x;
        v[4 * k + 1] += f.y;
        v[4 * k + 2] += f.z;
        v[4 * k + 3] += f.w;
      }
    }
    if (t < p.n) {
      // the 16 columns lie wholly in a (c0 < h_v) or in b: h_v is a multiple of 16
      const int c0 = 16 * g;
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(c0 < p.h_v ? p.a : p.b) +
                           t * p.h_v + (c0 < p.h_v ? c0 : c0 - p.h_v);
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
  // Only this CTA's own shared memory is written by the others, and all of
  // that has landed: it may exit without waiting for the rest of the cluster.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

// Tensor map of a row-major [rows][cols] bf16 matrix: boxes of 64 columns x
// box_rows rows, 128-byte swizzle (the K-major operand layout of the MMA),
// zero fill outside the matrix.
static cudaError_t make_map(CUtensorMap* map, const void* ptr, int64_t cols, int64_t rows,
                            uint32_t box_rows) {
  const auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(gdn_tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)KB, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace proj
}  // namespace gdn

// The caller has checked: n > 0, d_model a positive multiple of 64, h_v a
// multiple of 16 with 2 h_v <= 256, every pointer 16-byte aligned.
cudaError_t gdn_launch_gate_projection(const void* hidden, const void* w_ba, int d_model,
                                       int64_t n, int h_v, void* a, void* b, int32_t* d_status,
                                       cudaStream_t s) {
  using namespace gdn::proj;
  cudaError_t e = cudaSuccess;
  CUtensorMap hmap, wmap;
  if ((e = make_map(&hmap, hidden, d_model, n, TM)) != cudaSuccess) return e;
  if ((e = make_map(&wmap, w_ba, d_model, 2 * h_v, (uint32_t)(2 * h_v))) != cudaSuccess) return e;
  ProjArgs p;
  p.a = a;
  p.b = b;
  p.d_status = d_status;
  p.n = n;
  p.h_v = h_v;
  p.nkb = d_model / KB;
  p.split = p.nkb < MAX_SPLIT ? (p.nkb >= 2 ? 2 : 1) : MAX_SPLIT;
  const uint32_t stage_bytes = A_BYTES + (uint32_t)(2 * h_v) * KB * 2;
  const int per_rank = (p.nkb + p.split - 1) / p.split;
  // the pushed partials: (split - 1) sources x groups per rank x 128 rows
  const int G = 2 * h_v / 16, gpr = (G + p.split - 1) / p.split;
  const uint32_t slot_bytes = (uint32_t)((p.split - 1) * gpr * TM) * SLOT_ROW;
  int stages = (int)((SMEM_BYTES - slot_bytes) / stage_bytes);
  if (stages > MAX_STAGES) stages = MAX_STAGES;
  if (stages > per_rank) stages = per_rank;
  if (stages < 1) return cudaErrorInvalidValue;   // not reached for 2 h_v <= 256
  p.stages = stages;
  p.slots = (uint32_t)stages * stage_bytes;
  p.wait_ns = 4000000000ull;
  const int smem = (int)(p.slots + slot_bytes) + 1024;
  // the shared-memory opt-in once per device (the largest size any shape uses)
  static int opted_in[64] = {};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !opted_in[dev]) {
    if ((e = cudaFuncSetAttribute(gate_projection_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)SMEM_BYTES + 1024)) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < 64) opted_in[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + TM - 1) / TM), (unsigned)p.split, 1);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)p.split;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gate_projection_kernel, p, hmap, wmap);
}
