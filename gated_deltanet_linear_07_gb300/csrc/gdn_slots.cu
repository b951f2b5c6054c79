// gdn_slots.cu -- copies of whole recurrent slots: the fp32 state and the conv
// window of slot src[i] to slot dst[i].  Snapshot (a live slot to a spare one),
// restore (back) and fork (one prefix into several sequences) are all this copy
// (Vallmo.jl README, src/: recurrent state snapshotted and restored for prefix
// caching; PicoLM changelog, SSM State Checkpointing: capture / restore the
// full SSM state).
//
// HBM-bound: each pair reads and writes state_bytes + window_bytes.  Grid
// (blocks per pair, pairs); each block copies 16-byte pieces with a grid-stride
// loop over the pair's two ranges, streaming loads and stores.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int COPY_THREADS = 256;
constexpr int PIECES_PER_THREAD = 4;

__global__ void __launch_bounds__(COPY_THREADS) slot_copy_kernel(
    float* __restrict__ state_pool, unsigned char* __restrict__ conv_pool, int64_t num_slots,
    int64_t state_pieces, int64_t window_pieces, const int32_t* __restrict__ src,
    const int32_t* __restrict__ dst, int32_t* d_status) {
  const int p = blockIdx.y;
  const int32_t s = src[p], d = dst[p];
  if (s < 0 || d < 0) return;                      // padding pair
  if (s >= num_slots || d >= num_slots) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(d_status, GDN_DEV_BAD_SLOT);
    return;
  }
  if (s == d) return;
  const uint4* st_src = reinterpret_cast<const uint4*>(state_pool) + (size_t)s * state_pieces;
  uint4* st_dst = reinterpret_cast<uint4*>(state_pool) + (size_t)d * state_pieces;
  const uint4* w_src = reinterpret_cast<const uint4*>(conv_pool) + (size_t)s * window_pieces;
  uint4* w_dst = reinterpret_cast<uint4*>(conv_pool) + (size_t)d * window_pieces;
  const int64_t total = state_pieces + window_pieces;
  const int64_t stride = (int64_t)gridDim.x * COPY_THREADS;
  for (int64_t i = (int64_t)blockIdx.x * COPY_THREADS + threadIdx.x; i < total; i += stride) {
    if (i < state_pieces) __stcs(st_dst + i, __ldcs(st_src + i));
    else __stcs(w_dst + (i - state_pieces), __ldcs(w_src + (i - state_pieces)));
  }
}

}  // namespace
}  // namespace gdn

cudaError_t gdn_launch_slot_copy(float* state_pool, void* conv_pool, int64_t num_slots,
                                 int64_t state_bytes, int64_t window_bytes, const int32_t* src,
                                 const int32_t* dst, int32_t n, int32_t* d_status,
                                 cudaStream_t s) {
  using namespace gdn;
  if (n <= 0) return cudaSuccess;
  const int64_t sp = state_bytes / 16, wp = window_bytes / 16;
  const int64_t per_block = (int64_t)COPY_THREADS * PIECES_PER_THREAD;
  const int64_t bx = (sp + wp + per_block - 1) / per_block;
  // gridDim.y is at most 65535 pairs per launch
  for (int32_t first = 0; first < n; first += 65535) {
    const int32_t cnt = n - first < 65535 ? n - first : 65535;
    slot_copy_kernel<<<dim3((unsigned)bx, (unsigned)cnt), COPY_THREADS, 0, s>>>(
        state_pool, reinterpret_cast<unsigned char*>(conv_pool), num_slots, sp, wp, src + first,
        dst + first, d_status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
