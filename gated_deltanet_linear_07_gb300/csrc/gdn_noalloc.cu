// gdn_noalloc.cu -- gdn_prefill_noalloc: the prefill for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc: code embedded in a host framework or
// serving engine whose allocator has already reserved (nearly) all of HBM for
// its own caches and pools, and hot paths where the implicit device-wide
// synchronisation that cudaMalloc/cudaFree may perform is not acceptable.
// gdn_prefill needs a workspace they would have to allocate; this entry point
// uses a fixed scratch array that lives in the library's own device image
// instead.  The caller still passes every input and output buffer.
//
// The scratch is GDN_NOALLOC_SCRATCH_BYTES of file-scope __device__ memory:
// every GPU that loads this library holds it until the process exits.  Host
// code only ever sees a host-side stand-in under that name, never a device
// address, so the device address is looked up once per device (with that
// device current) by cudaGetSymbolAddress, cached, and handed to the kernels.
#include <mutex>

#include "gdn_common.cuh"

#define GDN_EXPORT extern "C" __attribute__((visibility("default")))

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_setup_mu;
void* g_scratch_dev[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device; the first call
// on a device does the lookup.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ECUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return GDN_ECUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return GDN_OK;
}

}  // namespace

GDN_EXPORT int gdn_prefill_noalloc(const gdn_dims* dims, const gdn_params* params,
                                   const void* x, const void* a, const void* b,
                                   const int32_t* cu_seqlens, int32_t num_seqs,
                                   int64_t total_tokens, const int32_t* slot_idx,
                                   const uint8_t* has_initial_state, float* state_pool,
                                   void* conv_pool, int64_t num_slots, void* o,
                                   int32_t* d_status, gdn_stream_t stream) {
  const size_t need = gdn_prefill_workspace_size(dims, total_tokens, num_seqs);
  if (need == 0)  // bad dimensions or sizes: let gdn_prefill name the problem
    return gdn_prefill(dims, params, x, a, b, cu_seqlens, num_seqs, total_tokens, slot_idx,
                       has_initial_state, state_pool, conv_pool, num_slots, o, nullptr, 0,
                       d_status, stream);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_EWORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != GDN_OK) return rc;
  // Nothing in the scratch has to start at zero: every kernel writes each
  // workspace word before any kernel reads it.
  return gdn_prefill(dims, params, x, a, b, cu_seqlens, num_seqs, total_tokens, slot_idx,
                     has_initial_state, state_pool, conv_pool, num_slots, o, scratch,
                     (size_t)GDN_NOALLOC_SCRATCH_BYTES, d_status, stream);
}
