// gdn_check.cu -- row and state scans of the GDN_CHECK_FINITE probe
// (gdn_check.cuh).  A value is non-finite when its exponent bits are all ones.
#include "gdn_check.cuh"

namespace gdn {
namespace {

constexpr int CHECK_THREADS = 128;

__device__ __forceinline__ bool bad_f32(uint32_t u) { return (u & 0x7f800000u) == 0x7f800000u; }
__device__ __forceinline__ bool bad_bf16(uint32_t u) { return (u & 0x7f80u) == 0x7f80u; }

// Sequence of row t: the largest b with cu[b] <= t (skips empty sequences).
__device__ __forceinline__ int seq_of_row(const int32_t* __restrict__ cu, int num_seqs, int64_t t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(CHECK_THREADS) check_rows_kernel(const GdnPrefillArgs a,
                                                                   const void* p, int bf16,
                                                                   int64_t row_elems, int bit) {
  if (!a.ws_flag[0]) return;
  const int64_t t = blockIdx.x;
  const int slot = a.slot_idx[seq_of_row(a.cu_seqlens, a.num_seqs, t)];
  if (slot < 0 || slot >= a.num_slots) return;
  bool bad = false;
  if (bf16) {
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p) + t * row_elems;
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x) bad |= bad_bf16(q[e]);
  } else {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p) + t * row_elems;
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x) bad |= bad_f32(q[e]);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(a.d_status, bit);
}

__global__ void __launch_bounds__(CHECK_THREADS) check_states_kernel(const GdnPrefillArgs a,
                                                                     int64_t elems, int bit) {
  if (!a.ws_flag[0]) return;
  const int b = blockIdx.x, h = blockIdx.y;
  const int slot = a.slot_idx[b];
  if (slot < 0 || slot >= a.num_slots) return;
  const uint32_t* st =
      reinterpret_cast<const uint32_t*>(a.state_pool) + ((size_t)slot * a.h_v + h) * elems;
  bool bad = false;
  for (int64_t e = threadIdx.x; e < elems; e += blockDim.x) bad |= bad_f32(st[e]);
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(a.d_status, bit);
}

}  // namespace
}  // namespace gdn

cudaError_t gdn_check_rows(const GdnPrefillArgs& a, const void* p, bool bf16, int64_t row_elems,
                           int bit, cudaStream_t s) {
  if (a.total_tokens == 0 || row_elems == 0) return cudaSuccess;
  gdn::check_rows_kernel<<<(unsigned)a.total_tokens, gdn::CHECK_THREADS, 0, s>>>(
      a, p, bf16 ? 1 : 0, row_elems, bit);
  return cudaGetLastError();
}

cudaError_t gdn_check_states(const GdnPrefillArgs& a, int d_k, int d_v, int bit, cudaStream_t s) {
  if (a.num_seqs == 0) return cudaSuccess;
  gdn::check_states_kernel<<<dim3(a.num_seqs, a.h_v), gdn::CHECK_THREADS, 0, s>>>(
      a, (int64_t)d_k * d_v, bit);
  return cudaGetLastError();
}
