// gdn_api.cu -- the C ABI declared in include/gdn.h: host-side argument
// checks, workspace carve-up and kernel dispatch.  Nothing here allocates,
// synchronises or keeps state between calls.
#include <stdint.h>
#include <string.h>

#include "gdn_check.cuh"
#include "gdn_common.cuh"

#define GDN_EXPORT extern "C" __attribute__((visibility("default")))

size_t gdn_simt_scan_smem_bytes(int chunk, int d_k, int d_v);

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kMaxSmem = 227 * 1024;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool pow2_dim(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t conv_dim_of(const gdn_dims* d) {
  return 2 * (int64_t)d->h_k * d->d_k + (int64_t)d->h_v * d->d_v;
}

int check_dims(const gdn_dims* d) {
  if (!d) return GDN_EINVAL;
  if (d->h_k <= 0 || d->h_v <= 0 || d->h_v % d->h_k != 0) return GDN_EINVAL;
  if (!(d->l2_eps >= 0.0f)) return GDN_EINVAL;
  if (d->flags & ~(GDN_FP32_STATE | GDN_CHECK_FINITE | GDN_TEST_WAIT_TIMEOUT | GDN_BF16_OPERANDS))
    return GDN_EINVAL;
  if (!pow2_dim(d->d_k) || !pow2_dim(d->d_v)) return GDN_EUNSUPPORTED;
  if (d->conv_w != 4) return GDN_EUNSUPPORTED;
  if (d->io != GDN_FP32 && d->io != GDN_BF16) return GDN_EUNSUPPORTED;
  if (d->h_k > 65535 || d->h_v > 65535) return GDN_EUNSUPPORTED;   // grid y extents
  // the prefill front end stages one token's conv output in shared memory
  if (conv_dim_of(d) * (int64_t)sizeof(float) > (int64_t)kMaxSmem) return GDN_EUNSUPPORTED;
  return GDN_OK;
}

int check_prefill_dims(const gdn_dims* d) {
  int rc = check_dims(d);
  if (rc != GDN_OK) return rc;
  if (d->chunk != 16 && d->chunk != 32 && d->chunk != 64 && d->chunk != 128) return GDN_EUNSUPPORTED;
  // the SIMT path keeps a chunk's factors in shared memory (it streams the scan's
  // inputs and narrows its d_v tile where they would not fit)
  if (gdn_simt_scan_smem_bytes(d->chunk, d->d_k, d->d_v) > kMaxSmem) return GDN_EUNSUPPORTED;
  return GDN_OK;
}

// The tensor-core path, for its shapes, when there are tokens.  A call whose
// sequences are all empty has only states and windows to pass through (or to
// zero): the SIMT path's check, window write-back and scan do exactly that
// and build no tensor map over an x with no rows.
bool use_tc(const gdn_dims* d, int64_t total_tokens) {
  return total_tokens > 0 && (d->flags & GDN_FP32_STATE) == 0 &&
         gdn_tc_prefill_supported(d->h_k, d->h_v, d->d_k, d->d_v, d->chunk, d->io);
}

struct PrefillLayout {
  // SIMT path
  size_t flag, q, k, v, g, beta, u, wk, p, gam;
  // tensor-core path
  size_t chunk_off, ready, kq, vh;
  int64_t max_chunks;
  size_t total;
};

PrefillLayout prefill_layout(const gdn_dims* d, int64_t T, int64_t B) {
  PrefillLayout L;
  memset(&L, 0, sizeof(L));
  size_t o = 0;
  L.flag = o; o += align_up(16);
  if (use_tc(d, T)) {
    L.max_chunks = (T + d->chunk - 1) / d->chunk + B;
    L.chunk_off = o; o += align_up((size_t)(B + 1) * sizeof(int32_t));
    L.ready = o; o += align_up((size_t)L.max_chunks * d->h_k * sizeof(int32_t));
    o = (o + 1023) / 1024 * 1024;
    L.kq = o; o += (size_t)L.max_chunks * d->h_k * gdn_tc_kq_bytes();
    L.vh = o; o += (size_t)L.max_chunks * d->h_v * gdn_tc_vh_bytes();
  } else {
    L.max_chunks = (T + d->chunk - 1) / d->chunk + B;
    L.chunk_off = o; o += align_up((size_t)(B + 1) * sizeof(int32_t));
    L.q = o; o += align_up((size_t)T * d->h_k * d->d_k * sizeof(float));
    L.k = o; o += align_up((size_t)T * d->h_k * d->d_k * sizeof(float));
    L.v = o; o += align_up((size_t)T * d->h_v * d->d_v * sizeof(float));
    L.g = o; o += align_up((size_t)T * d->h_v * sizeof(float));
    L.beta = o; o += align_up((size_t)T * d->h_v * sizeof(float));
    L.u = o; o += align_up((size_t)T * d->h_v * d->d_v * sizeof(float));
    L.wk = o; o += align_up((size_t)T * d->h_v * d->d_k * sizeof(float));
    L.p = o; o += align_up((size_t)T * d->h_v * d->chunk * sizeof(float));
    L.gam = o; o += align_up((size_t)T * d->h_v * sizeof(float));
  }
  L.total = o;
  return L;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ECUDA; }

}  // namespace

GDN_EXPORT const char* gdn_status_str(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_EINVAL: return "invalid argument";
    case GDN_EUNSUPPORTED: return "unsupported dimensions";
    case GDN_ECUDA: return "CUDA launch or runtime error";
    case GDN_EWORKSPACE: return "workspace missing or too small";
    case GDN_EALIGN: return "device pointer not 16-byte aligned";
  }
  return "unknown status";
}

GDN_EXPORT int gdn_conv1d_update(const gdn_dims* dims, const float* conv_weight,
                                 const void* x, void* conv_pool, int64_t num_slots,
                                 const int32_t* slot_idx, int32_t n, void* y,
                                 int32_t* d_status, gdn_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != GDN_OK) return rc;
  if (n < 0 || num_slots < 0) return GDN_EINVAL;
  if (n == 0) return GDN_OK;
  if (!conv_weight || !x || !conv_pool || !slot_idx || !y) return GDN_EINVAL;
  if (!aligned16(conv_weight) || !aligned16(conv_pool)) return GDN_EALIGN;
  GdnConvArgs a;
  a.conv_dim = (int32_t)conv_dim_of(dims);
  a.conv_w = dims->conv_w;
  a.n = n;
  a.num_slots = num_slots;
  a.x = x;
  a.slot_idx = slot_idx;
  a.conv_weight = conv_weight;
  a.conv_pool = conv_pool;
  a.y = y;
  a.d_status = d_status;
  return cuda_rc(gdn_launch_conv_update(a, dims->io, reinterpret_cast<cudaStream_t>(stream)));
}

GDN_EXPORT int gdn_gated_rmsnorm(const gdn_dims* dims, const float* weight, float eps,
                                 const void* o, const void* z, int64_t n, void* y,
                                 gdn_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != GDN_OK) return rc;
  if (n < 0 || !(eps >= 0.f)) return GDN_EINVAL;
  if (dims->d_v != 16 && dims->d_v != 32 && dims->d_v != 64 && dims->d_v != 128)
    return GDN_EUNSUPPORTED;
  if (n == 0) return GDN_OK;
  if (!weight || !o || !z || !y) return GDN_EINVAL;
  if (!aligned16(weight) || !aligned16(o) || !aligned16(z) || !aligned16(y)) return GDN_EALIGN;
  return cuda_rc(gdn_launch_gated_rmsnorm(weight, eps, o, z, n * dims->h_v, dims->d_v, dims->io, y,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

GDN_EXPORT int gdn_gate_projection(const gdn_dims* dims, const void* hidden, const void* w_ba,
                                   int32_t d_model, int64_t n, void* a, void* b,
                                   int32_t* d_status, gdn_stream_t stream) {
  if (!dims || n < 0 || d_model <= 0) return GDN_EINVAL;
  if (dims->h_v <= 0) return GDN_EINVAL;
  if (dims->h_v % 16 != 0 || 2 * dims->h_v > 256 || d_model % 64 != 0) return GDN_EUNSUPPORTED;
  if (n > (int64_t)INT32_MAX) return GDN_EUNSUPPORTED;   // 128-token tiles index the grid
  if (n == 0) return GDN_OK;
  if (!hidden || !w_ba || !a || !b) return GDN_EINVAL;
  if (!aligned16(hidden) || !aligned16(w_ba) || !aligned16(a) || !aligned16(b)) return GDN_EALIGN;
  return cuda_rc(gdn_launch_gate_projection(hidden, w_ba, d_model, n, dims->h_v, a, b, d_status,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

GDN_EXPORT size_t gdn_prefill_workspace_size(const gdn_dims* dims, int64_t total_tokens,
                                             int32_t num_seqs) {
  if (check_prefill_dims(dims) != GDN_OK || total_tokens < 0 || num_seqs < 0) return 0;
  return prefill_layout(dims, total_tokens, num_seqs).total;
}

// GDN_CHECK_FINITE: scans of what each stage of the call wrote (gdn_check.cuh).
static cudaError_t check_stages(const GdnPrefillArgs& p, const gdn_dims* d, bool tc,
                                cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  auto rows = [&](const void* ptr, bool bf16, int64_t n, int bit) {
    if (e == cudaSuccess) e = gdn_check_rows(p, ptr, bf16, n, bit, s);
  };
  if (tc) {
    e = gdn_check_tc_records(p, s);
  } else {
    rows(p.ws_q, false, (int64_t)d->h_k * d->d_k, GDN_DEV_NONFINITE_FRONTEND);
    rows(p.ws_k, false, (int64_t)d->h_k * d->d_k, GDN_DEV_NONFINITE_FRONTEND);
    rows(p.ws_v, false, (int64_t)d->h_v * d->d_v, GDN_DEV_NONFINITE_FRONTEND);
    rows(p.ws_g, false, d->h_v, GDN_DEV_NONFINITE_FRONTEND);
    rows(p.ws_beta, false, d->h_v, GDN_DEV_NONFINITE_FRONTEND);
    rows(p.ws_u, false, (int64_t)d->h_v * d->d_v, GDN_DEV_NONFINITE_CHUNK);
    rows(p.ws_wk, false, (int64_t)d->h_v * d->d_k, GDN_DEV_NONFINITE_CHUNK);
    rows(p.ws_p, false, (int64_t)d->h_v * d->chunk, GDN_DEV_NONFINITE_CHUNK);
    rows(p.ws_gam, false, d->h_v, GDN_DEV_NONFINITE_CHUNK);
  }
  rows(p.o, d->io == GDN_BF16, (int64_t)d->h_v * d->d_v, GDN_DEV_NONFINITE_OUT);
  if (e == cudaSuccess) e = gdn_check_states(p, d->d_k, d->d_v, GDN_DEV_NONFINITE_OUT, s);
  return e;
}

// The prefill behind every public variant; ckpt_every_chunks = 0 and
// ckpt_slot = null: no interval checkpoints.
static int prefill_impl(const gdn_dims* dims, const gdn_params* params, const void* x,
                        const void* a, const void* b, const int32_t* cu_seqlens, int32_t num_seqs,
                        int64_t total_tokens, const int32_t* slot_idx,
                        const uint8_t* has_initial_state, float* state_pool, void* conv_pool,
                        int64_t num_slots, void* o, void* workspace, size_t workspace_bytes,
                        int32_t ckpt_every_chunks, const int32_t* ckpt_slot, const void* z,
                        const float* norm_weight, float norm_eps, int32_t* d_status,
                        gdn_trace* trace, gdn_stream_t stream) {
  if (trace) {
    trace->launches = 0;
    trace->stages_run = 0;
  }
  int rc = check_prefill_dims(dims);
  if (rc != GDN_OK) return rc;
  if (!params || num_seqs < 0 || total_tokens < 0 || num_slots < 0) return GDN_EINVAL;
  const bool check_finite = (dims->flags & GDN_CHECK_FINITE) != 0;
  if (check_finite && !d_status) return GDN_EINVAL;   // the probe reports through it
  if (total_tokens > INT32_MAX) return GDN_EUNSUPPORTED;
  if (num_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_EINVAL;
  if (!params->conv_weight || !params->A_log || !params->dt_bias || !cu_seqlens || !slot_idx ||
      !state_pool || !conv_pool)
    return GDN_EINVAL;
  if (total_tokens > 0 && (!x || !a || !b || !o)) return GDN_EINVAL;
  if (!aligned16(params->conv_weight) || !aligned16(state_pool) || !aligned16(conv_pool) ||
      (x && !aligned16(x)) || (o && !aligned16(o)))
    return GDN_EALIGN;
  const PrefillLayout L = prefill_layout(dims, total_tokens, num_seqs);
  if (!workspace || workspace_bytes < L.total) return GDN_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return GDN_EALIGN;

  GdnPrefillArgs p;
  memset(&p, 0, sizeof(p));
  p.h_k = dims->h_k; p.h_v = dims->h_v; p.d_k = dims->d_k; p.d_v = dims->d_v;
  p.conv_w = dims->conv_w; p.chunk = dims->chunk;
  p.conv_dim = (int32_t)conv_dim_of(dims);
  p.num_seqs = num_seqs; p.total_tokens = total_tokens; p.num_slots = num_slots;
  p.l2_eps = dims->l2_eps;
  p.x = x; p.a = a; p.b = b;
  p.cu_seqlens = cu_seqlens; p.slot_idx = slot_idx; p.has_init = has_initial_state;
  p.conv_weight = params->conv_weight; p.A_log = params->A_log; p.dt_bias = params->dt_bias;
  p.state_pool = state_pool; p.conv_pool = conv_pool; p.o = o; p.d_status = d_status;
  p.ckpt_every_chunks = ckpt_every_chunks; p.ckpt_slot = ckpt_slot;
  // Waits between CTAs and warps give up after 4 s (a chunk takes microseconds);
  // the test knob shortens that to 2 ms and withholds one chunk's flag.
  const bool test_timeout = (dims->flags & GDN_TEST_WAIT_TIMEOUT) != 0;
  p.wait_ns = test_timeout ? 2000000ull : 4000000000ull;
  p.withhold_last_chunk = test_timeout ? 1 : 0;
  p.bf16_ops = (dims->flags & GDN_BF16_OPERANDS) != 0 ? 1 : 0;
  char* ws = reinterpret_cast<char*>(workspace);
  p.ws_flag = reinterpret_cast<int32_t*>(ws + L.flag);
  p.ws_q = reinterpret_cast<float*>(ws + L.q);
  p.ws_k = reinterpret_cast<float*>(ws + L.k);
  p.ws_v = reinterpret_cast<float*>(ws + L.v);
  p.ws_g = reinterpret_cast<float*>(ws + L.g);
  p.ws_beta = reinterpret_cast<float*>(ws + L.beta);
  cudaError_t e;
  const bool tc = use_tc(dims, total_tokens);
  if (tc) {
    p.chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_off);
    p.chunk_ready = reinterpret_cast<int32_t*>(ws + L.ready);
    p.max_chunks = L.max_chunks;
    p.kq_ws = reinterpret_cast<uint8_t*>(ws + L.kq);
    p.vh_ws = reinterpret_cast<uint8_t*>(ws + L.vh);
    e = gdn_launch_prefill_tc(p, reinterpret_cast<cudaStream_t>(stream), trace);
  } else {
    p.chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_off);
    p.max_chunks = L.max_chunks;
    p.ws_u = reinterpret_cast<float*>(ws + L.u);
    p.ws_wk = reinterpret_cast<float*>(ws + L.wk);
    p.ws_p = reinterpret_cast<float*>(ws + L.p);
    p.ws_gam = reinterpret_cast<float*>(ws + L.gam);
    e = gdn_launch_prefill_simt(p, dims->io, reinterpret_cast<cudaStream_t>(stream), trace);
  }
  // The gated norm of the output, in place on o, right after the layer: both
  // prefill scans write o from several warps or CTAs per token, and a norm in
  // the tensor-core scan's output warps lengthened its chunk period (they are
  // short of issue slots there), so the standalone kernel is the faster way.
  if (e == cudaSuccess && z && total_tokens > 0)
    e = gdn_launch_gated_rmsnorm(norm_weight, norm_eps, o, z, total_tokens * dims->h_v, dims->d_v,
                                 dims->io, o, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess && check_finite)
    e = check_stages(p, dims, tc, reinterpret_cast<cudaStream_t>(stream));
  return cuda_rc(e);
}

GDN_EXPORT int gdn_prefill_traced(const gdn_dims* dims, const gdn_params* params,
                                  const void* x, const void* a, const void* b,
                                  const int32_t* cu_seqlens, int32_t num_seqs,
                                  int64_t total_tokens, const int32_t* slot_idx,
                                  const uint8_t* has_initial_state, float* state_pool,
                                  void* conv_pool, int64_t num_slots, void* o, void* workspace,
                                  size_t workspace_bytes, int32_t* d_status, gdn_trace* trace,
                                  gdn_stream_t stream) {
  return prefill_impl(dims, params, x, a, b, cu_seqlens, num_seqs, total_tokens, slot_idx,
                      has_initial_state, state_pool, conv_pool, num_slots, o, workspace,
                      workspace_bytes, 0, nullptr, nullptr, nullptr, 0.f, d_status, trace, stream);
}

GDN_EXPORT int gdn_prefill_checkpointed(const gdn_dims* dims, const gdn_params* params,
                                        const void* x, const void* a, const void* b,
                                        const int32_t* cu_seqlens, int32_t num_seqs,
                                        int64_t total_tokens, const int32_t* slot_idx,
                                        const uint8_t* has_initial_state, float* state_pool,
                                        void* conv_pool, int64_t num_slots, void* o,
                                        void* workspace, size_t workspace_bytes,
                                        int64_t ckpt_every, const int32_t* ckpt_slot,
                                        int32_t* d_status, gdn_stream_t stream) {
  const int rc = check_prefill_dims(dims);   // validates chunk before the division below
  if (rc != GDN_OK) return rc;
  if (ckpt_every <= 0 || ckpt_every % dims->chunk != 0 || !ckpt_slot) return GDN_EINVAL;
  if (ckpt_every / dims->chunk > INT32_MAX) return GDN_EUNSUPPORTED;
  return prefill_impl(dims, params, x, a, b, cu_seqlens, num_seqs, total_tokens, slot_idx,
                      has_initial_state, state_pool, conv_pool, num_slots, o, workspace,
                      workspace_bytes, (int32_t)(ckpt_every / dims->chunk), ckpt_slot, nullptr,
                      nullptr, 0.f, d_status, nullptr, stream);
}

GDN_EXPORT int gdn_prefill_gated_norm(const gdn_dims* dims, const gdn_params* params,
                                      const void* x, const void* a, const void* b,
                                      const int32_t* cu_seqlens, int32_t num_seqs,
                                      int64_t total_tokens, const int32_t* slot_idx,
                                      const uint8_t* has_initial_state, float* state_pool,
                                      void* conv_pool, int64_t num_slots, const void* z,
                                      const float* norm_weight, float eps, void* y,
                                      void* workspace, size_t workspace_bytes, int32_t* d_status,
                                      gdn_stream_t stream) {
  const int rc = check_prefill_dims(dims);
  if (rc != GDN_OK) return rc;
  if (!(eps >= 0.f) || eps > 1e30f) return GDN_EINVAL;   // also rejects NaN
  if (total_tokens > 0 && (!z || !norm_weight)) return GDN_EINVAL;
  if (z && z == y) return GDN_EINVAL;   // the SIMT path writes o into y before the norm reads z
  if ((z && !aligned16(z)) || (norm_weight && !aligned16(norm_weight))) return GDN_EALIGN;
  return prefill_impl(dims, params, x, a, b, cu_seqlens, num_seqs, total_tokens, slot_idx,
                      has_initial_state, state_pool, conv_pool, num_slots, y, workspace,
                      workspace_bytes, 0, nullptr, total_tokens > 0 ? z : nullptr, norm_weight,
                      eps, d_status, nullptr, stream);
}

GDN_EXPORT int gdn_slot_copy(const gdn_dims* dims, float* state_pool, void* conv_pool,
                             int64_t num_slots, const int32_t* src_slot, const int32_t* dst_slot,
                             int32_t n, int32_t* d_status, gdn_stream_t stream) {
  const int rc = check_dims(dims);
  if (rc != GDN_OK) return rc;
  if (n < 0 || num_slots < 0) return GDN_EINVAL;
  if (n == 0) return GDN_OK;
  if (!state_pool || !conv_pool || !src_slot || !dst_slot) return GDN_EINVAL;
  if (!aligned16(state_pool) || !aligned16(conv_pool)) return GDN_EALIGN;
  const int64_t state_bytes = (int64_t)dims->h_v * dims->d_k * dims->d_v * 4;
  const int64_t window_bytes =
      (int64_t)(dims->conv_w - 1) * conv_dim_of(dims) * (dims->io == GDN_BF16 ? 2 : 4);
  if (state_bytes % 16 != 0 || window_bytes % 16 != 0) return GDN_EUNSUPPORTED;
  return cuda_rc(gdn_launch_slot_copy(state_pool, conv_pool, num_slots, state_bytes, window_bytes,
                                      src_slot, dst_slot, n, d_status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

GDN_EXPORT int gdn_prefill(const gdn_dims* dims, const gdn_params* params, const void* x,
                           const void* a, const void* b, const int32_t* cu_seqlens,
                           int32_t num_seqs, int64_t total_tokens, const int32_t* slot_idx,
                           const uint8_t* has_initial_state, float* state_pool,
                           void* conv_pool, int64_t num_slots, void* o, void* workspace,
                           size_t workspace_bytes, int32_t* d_status, gdn_stream_t stream) {
  return gdn_prefill_traced(dims, params, x, a, b, cu_seqlens, num_seqs, total_tokens, slot_idx,
                            has_initial_state, state_pool, conv_pool, num_slots, o, workspace,
                            workspace_bytes, d_status, nullptr, stream);
}

// The decode step behind both public variants; z = null: plain o.
static int decode_impl(const gdn_dims* dims, const gdn_params* params, const void* x,
                       const void* a, const void* b, const int32_t* slot_idx, int32_t n,
                       float* state_pool, void* conv_pool, int64_t num_slots, void* o,
                       const void* z, const float* norm_weight, float norm_eps,
                       int32_t* d_status, gdn_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != GDN_OK) return rc;
  if (!params || n < 0 || num_slots < 0) return GDN_EINVAL;
  if (n == 0) return GDN_OK;
  if (!params->conv_weight || !params->A_log || !params->dt_bias || !x || !a || !b ||
      !slot_idx || !state_pool || !conv_pool || !o)
    return GDN_EINVAL;
  if (!aligned16(params->conv_weight) || !aligned16(state_pool) || !aligned16(conv_pool) ||
      !aligned16(x) || !aligned16(o))
    return GDN_EALIGN;
  GdnDecodeArgs p;
  p.h_k = dims->h_k; p.h_v = dims->h_v;
  p.conv_dim = (int32_t)conv_dim_of(dims);
  p.n = n; p.l2_eps = dims->l2_eps; p.num_slots = num_slots;
  p.x = x; p.a = a; p.b = b; p.slot_idx = slot_idx;
  p.conv_weight = params->conv_weight; p.A_log = params->A_log; p.dt_bias = params->dt_bias;
  p.state_pool = state_pool; p.conv_pool = conv_pool; p.o = o; p.d_status = d_status;
  p.z = z; p.norm_weight = norm_weight; p.norm_eps = norm_eps;
  return cuda_rc(gdn_launch_decode(p, dims->d_k, dims->d_v, dims->io,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

GDN_EXPORT int gdn_decode_step(const gdn_dims* dims, const gdn_params* params, const void* x,
                               const void* a, const void* b, const int32_t* slot_idx, int32_t n,
                               float* state_pool, void* conv_pool, int64_t num_slots, void* o,
                               int32_t* d_status, gdn_stream_t stream) {
  return decode_impl(dims, params, x, a, b, slot_idx, n, state_pool, conv_pool, num_slots, o,
                     nullptr, nullptr, 0.f, d_status, stream);
}

GDN_EXPORT int gdn_decode_step_gated_norm(const gdn_dims* dims, const gdn_params* params,
                                          const void* x, const void* a, const void* b,
                                          const int32_t* slot_idx, int32_t n, float* state_pool,
                                          void* conv_pool, int64_t num_slots, const void* z,
                                          const float* norm_weight, float eps, void* y,
                                          int32_t* d_status, gdn_stream_t stream) {
  const int rc = check_dims(dims);
  if (rc != GDN_OK) return rc;
  if (!(eps >= 0.f) || eps > 1e30f) return GDN_EINVAL;   // also rejects NaN
  if (n > 0 && (!z || !norm_weight)) return GDN_EINVAL;
  if (z && z == y) return GDN_EINVAL;
  if ((z && !aligned16(z)) || (norm_weight && !aligned16(norm_weight))) return GDN_EALIGN;
  return decode_impl(dims, params, x, a, b, slot_idx, n, state_pool, conv_pool, num_slots, y,
                     n > 0 ? z : nullptr, norm_weight, eps, d_status, stream);
}
