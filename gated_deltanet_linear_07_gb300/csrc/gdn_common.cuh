// gdn_common.cuh -- element I/O, gate math and small device helpers shared by
// the Gated DeltaNet kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// ---- element I/O --------------------------------------------------------

template <typename T>
__device__ __forceinline__ float ld_io(const T* p);
template <>
__device__ __forceinline__ float ld_io<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_io<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void st_io(T* p, float v);
template <>
__device__ __forceinline__ void st_io<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_io<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// Raw copy of one element (window roll: the stored inputs stay bit-exact).
template <typename T>
__device__ __forceinline__ void copy_io(T* dst, const T* src) { *dst = *src; }

// ---- gate and activation math (fp32, CUDA math library calls) -------------

// SiLU(z) = z * sigmoid(z)
__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// softplus(z) = log(1 + e^z) = max(z, 0) + log1p(e^{-|z|})
__device__ __forceinline__ float softplusf_(float z) {
  return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z)));
}

// g = -exp(A_log) * softplus(a + dt_bias)   (log-decay, <= 0)
__device__ __forceinline__ float gate_g(float a, float A_log, float dt_bias) {
  return -expf(A_log) * softplusf_(a + dt_bias);
}

__device__ __forceinline__ void set_status(int32_t* d_status, int bits) {
  if (d_status) atomicOr(d_status, bits);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Streaming (evict-first) 128-bit accesses for data touched exactly once.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

}  // namespace gdn

// Host-side launch descriptors shared between the API translation unit and
// the kernel translation units.
struct GdnDecodeArgs {
  int32_t h_k, h_v, conv_dim, n;
  float l2_eps;
  int64_t num_slots;
  const void* x;
  const void* a;
  const void* b;
  const int32_t* slot_idx;
  const float* conv_weight;
  const float* A_log;
  const float* dt_bias;
  float* state_pool;
  void* conv_pool;
  void* o;
  int32_t* d_status;
  // fused gated RMSNorm of the output (null z: plain o): o <- rmsnorm(o) w SiLU(z)
  const void* z;            // [n][h_v][d_v], I/O dtype
  const float* norm_weight; // [d_v]
  float norm_eps;
};

struct GdnConvArgs {
  int32_t conv_dim, conv_w, n;
  int64_t num_slots;
  const void* x;
  const int32_t* slot_idx;
  const float* conv_weight;
  void* conv_pool;
  void* y;
  int32_t* d_status;
};

struct GdnPrefillArgs {
  int32_t h_k, h_v, d_k, d_v, conv_w, chunk, conv_dim, num_seqs;
  int64_t total_tokens, num_slots;
  float l2_eps;
  const void* x;
  const void* a;
  const void* b;
  const int32_t* cu_seqlens;
  const int32_t* slot_idx;
  const uint8_t* has_init;
  const float* conv_weight;
  const float* A_log;
  const float* dt_bias;
  float* state_pool;
  void* conv_pool;
  void* o;
  int32_t* d_status;
  // workspace carve-up (device)
  int32_t* ws_flag;  // [0] = 1 when cu_seqlens is valid
  float* ws_q;       // [T][h_k][d_k] normalised, scaled queries
  float* ws_k;       // [T][h_k][d_k] normalised keys
  float* ws_v;       // [T][h_v][d_v]
  float* ws_g;       // [T][h_v] log-decay
  float* ws_beta;    // [T][h_v]
  // SIMT path, written by its chunk kernel per token row of each chunk
  float* ws_u;       // [T][h_v][d_v]  U = T diag(beta) V
  float* ws_wk;      // [T][h_v][d_k]  Wk = T diag(beta e^gamma) K
  float* ws_p;       // [T][h_v][chunk] P = tril(Q K^T * decay)
  float* ws_gam;     // [T][h_v]       cumulative log-decay inside the chunk
  // tensor-core path workspace
  int32_t* chunk_off;   // [num_seqs+1] first global chunk of each sequence
  int64_t max_chunks;   // bound on the number of chunks: ceil(T/64) + num_seqs
  uint8_t* kq_ws;       // [max_chunks][h_k] [K;Q] tile images
  uint8_t* vh_ws;       // [max_chunks][h_v] P | U^T | decay factors | Wk records
  int32_t* chunk_ready; // [max_chunks][h_k] set to 1 when the prep published the chunk
  // 1: the scan runs beside the prep and waits for each chunk's ready flag;
  // 0: the scan starts after the prep kernel has finished (no flags needed)
  int32_t publish;
  // every inter-CTA or inter-warp wait gives up after this many nanoseconds
  uint64_t wait_ns;
  // GDN_TEST_WAIT_TIMEOUT: the prep does not publish the last chunk of
  // sequence 0, key head 0 (the scan's wait for it runs out)
  int32_t withhold_last_chunk;
  // GDN_BF16_OPERANDS: bf16 instead of fp16 tensor-core operands
  int32_t bf16_ops;
  // interval checkpoints (0 / null: none): every ckpt_every_chunks chunks strictly
  // inside sequence b, the state and window go to slot ckpt_slot[b] + k - 1
  int32_t ckpt_every_chunks;
  const int32_t* ckpt_slot;   // [num_seqs], < 0: no checkpoints for that sequence
};

// Slot of checkpoint k >= 1 (after k * every chunks) of sequence b, or -1 when
// there is none there; out-of-range slots set the status bit and give -1.
__device__ __forceinline__ int64_t ckpt_slot_of(const GdnPrefillArgs& a, int b, int64_t chunks_done,
                                                int64_t seq_len) {
  if (a.ckpt_every_chunks <= 0 || chunks_done % a.ckpt_every_chunks != 0) return -1;
  if (chunks_done * a.chunk >= seq_len) return -1;
  const int32_t base = a.ckpt_slot[b];
  if (base < 0) return -1;
  const int64_t cs = (int64_t)base + chunks_done / a.ckpt_every_chunks - 1;
  if (cs >= a.num_slots) {
    gdn::set_status(a.d_status, GDN_DEV_BAD_SLOT);
    return -1;
  }
  return cs;
}

// Launchers (defined in the kernel translation units); return cudaError_t.
cudaError_t gdn_launch_decode(const GdnDecodeArgs& a, int d_k, int d_v, int io,
                              cudaStream_t s);
cudaError_t gdn_launch_conv_update(const GdnConvArgs& a, int io, cudaStream_t s);
cudaError_t gdn_launch_slot_copy(float* state_pool, void* conv_pool, int64_t num_slots,
                                 int64_t state_bytes, int64_t window_bytes, const int32_t* src,
                                 const int32_t* dst, int32_t n, int32_t* d_status,
                                 cudaStream_t s);
cudaError_t gdn_launch_gated_rmsnorm(const float* weight, float eps, const void* o, const void* z,
                                     int64_t rows, int d_v, int io, void* y, cudaStream_t s);
cudaError_t gdn_launch_prefill_simt(const GdnPrefillArgs& a, int io, cudaStream_t s,
                                    gdn_trace* trace);

cudaError_t gdn_launch_prefill_tc(const GdnPrefillArgs& a, cudaStream_t s, gdn_trace* trace);
// Pieces of the prefill shared by both paths (defined with the SIMT path).
cudaError_t gdn_launch_check(const GdnPrefillArgs& a, cudaStream_t s, gdn_trace* trace);
cudaError_t gdn_launch_window(const GdnPrefillArgs& a, int io, cudaStream_t s, gdn_trace* trace);
bool gdn_tc_prefill_supported(int h_k, int h_v, int d_k, int d_v, int chunk, int io);
// cuTensorMapEncodeTiled (the driver's, as a PFN_cuTensorMapEncodeTiled_v12000)
// looked up once through the runtime's entry-point query; null if unavailable.
void* gdn_tensor_map_encoder();
cudaError_t gdn_launch_gate_projection(const void* hidden, const void* w_ba, int d_model,
                                       int64_t n, int h_v, void* a, void* b, int32_t* d_status,
                                       cudaStream_t s);
size_t gdn_tc_kq_bytes();
size_t gdn_tc_vh_bytes();

// Stage-trace helpers: record the caller's event (if any) on the stream.
inline cudaError_t gdn_trace_mark(gdn_trace* tr, int stage, bool begin, cudaStream_t s) {
  if (!tr) return cudaSuccess;
  tr->stages_run |= 1 << stage;
  void* ev = begin ? tr->begin[stage] : tr->end[stage];
  return ev ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), s) : cudaSuccess;
}
inline void gdn_trace_count(gdn_trace* tr, int n) {
  if (tr) tr->launches += n;
}
