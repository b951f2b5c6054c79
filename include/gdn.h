/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet linear-attention library.
 *
 * The layer (per sequence b, value head h, token t):
 *   1. causal width-W conv over the mixed q|k|v channels, the W-1 previous raw
 *      inputs coming from a rolling per-sequence window, then SiLU
 *      (Vallmo README, "What's here": causal conv1d; oxydllm 0.0.0-alpha.12.2
 *      release notes, New Features, "Gated DeltaNet runtime": the causal-conv
 *      window kept in the sequence's slot);
 *   2. split into q (H_k heads of d_k), k (H_k x d_k), v (H_v x d_v),
 *      head-major; value head h uses key head h / (H_v/H_k); q and k are L2
 *      normalised (eps inside the root) and q is scaled by 1/sqrt(d_k)
 *      (PicoLM changelog, "GPU: Device-Native Pipeline Rewrite": conv1d,
 *      l2norm, head_permute kernels);
 *   3. gates g = -exp(A_log[h]) * softplus(a + dt_bias[h]) and
 *      beta = sigmoid(b) (oxydllm notes, New Features: ssm_a holds the
 *      negated exponential of A_log; the scalars stay F32);
 *   4. the gated delta rule on a d_v x d_k fp32 memory S:
 *        S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *        o_t = S_t q_t
 *      (Gated DeltaNet, named as prior art in the valkyr README's License
 *      section; the 32x128x128 F32 memory, the chunked parallel scan for
 *      prefill and the O(1) recurrent step for decode are in the oxydllm
 *      notes, New Features, "Gated DeltaNet runtime").
 *
 * Memory layouts (row-major; "IO" is the element type named by gdn_dims.io):
 *   x            [rows][conv_dim] IO, conv_dim = 2*h_k*d_k + h_v*d_v,
 *                channels ordered q | k | v, each head-major
 *   a, b         [rows][h_v] IO
 *   o            [rows][h_v][d_v] IO
 *   conv_weight  [conv_dim][conv_w] fp32; tap conv_w-1 multiplies the newest
 *                input
 *   A_log, dt_bias [h_v] fp32
 *   state_pool   [num_slots][h_v][d_k][d_v] fp32: S stored transposed, so the
 *                value index is contiguous
 *   conv_pool    [num_slots][conv_w-1][conv_dim] IO: the last conv_w-1 raw
 *                inputs of the slot's sequence, oldest row first
 *
 * Ownership and threading: the caller owns every buffer; all data pointers
 * are DEVICE pointers except the dims/params structs, which are read on the
 * host during the call.  The library allocates no device memory, keeps no
 * mutable global state, never synchronises the stream and returns as soon as
 * the work is enqueued on `stream`.  Calls on different streams that touch
 * different slots may run concurrently.  Because a call only enqueues kernels
 * on `stream`, it can be captured into a CUDA graph and replayed; a replay
 * reuses the pointers, sizes and dimensions of the captured call (the first
 * gdn_prefill_noalloc call on a device must come before any capture).
 *
 * Errors: a negative gdn_status is returned synchronously for anything the
 * host can check (null pointers, unsupported dimensions, misalignment, a
 * workspace that is too small, a failed launch); nothing is enqueued then.
 * Problems only the device can see set bits in *d_status (optional device
 * int32, OR-ed, never cleared by the library; read it after the stream
 * synchronises) and the affected row or sequence is skipped.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum {
  GDN_OK = 0,
  GDN_EINVAL = -1,        /* null pointer, negative size, bad cu_seqlens count */
  GDN_EUNSUPPORTED = -2,  /* dimensions this build has no kernel for */
  GDN_ECUDA = -3,         /* a CUDA launch or runtime call failed */
  GDN_EWORKSPACE = -4,    /* workspace null or smaller than required */
  GDN_EALIGN = -5         /* a device pointer is not 16-byte aligned */
} gdn_status;

typedef enum { GDN_FP32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Bits of *d_status. */
#define GDN_DEV_BAD_SLOT 0x1        /* slot index out of range (prefill: < 0 or >= num_slots;
                                       decode: >= num_slots): row/sequence skipped */
#define GDN_DEV_BAD_CU_SEQLENS 0x2  /* cu_seqlens not 0..total_tokens non-decreasing: call skipped */
#define GDN_DEV_WAIT_TIMEOUT 0x4    /* an inter-CTA wait gave up: results invalid */
/* With GDN_CHECK_FINITE (prefill): a NaN or Inf among what the stage wrote. */
#define GDN_DEV_NONFINITE_FRONTEND 0x8  /* the front end's q, k (and v, gates on the SIMT path) */
#define GDN_DEV_NONFINITE_CHUNK 0x10    /* the chunk factors: P, U, Wk, decays */
#define GDN_DEV_NONFINITE_OUT 0x20      /* the layer output o (y) or a final state */

/* Bits of gdn_dims.flags.
 * GDN_FP32_STATE: prefill keeps every product with the fp32 state in fp32
 *   arithmetic (the SIMT path, any supported shape and chunk).  Without it the
 *   tensor-core path, where it applies (d_k = d_v = 128, chunk 64, bf16 I/O,
 *   h_v = 2 h_k), feeds the state and every other MMA operand to the tensor
 *   cores rounded to fp16 (10-bit mantissa; products accumulate in fp32), so
 *   its operands must stay within fp16 range (|value| < 65504: normalised
 *   q, k, the gates' factors, v = SiLU(conv(x)) and the state, all far below
 *   that for realistic activations); the error that rounding leaves in the
 *   state and in o is measured against the fp32 option on long,
 *   correlated-key sequences by the precision tests.  Decode always uses
 *   fp32 state products. */
#define GDN_FP32_STATE 0x1
/* GDN_CHECK_FINITE: after a prefill call (any prefill entry point) the library
 *   scans what each stage wrote -- its workspace records or rows, the output,
 *   the final states of the sequences with a valid slot -- and ORs
 *   GDN_DEV_NONFINITE_FRONTEND / _CHUNK / _OUT into *d_status for each stage
 *   that produced a NaN or Inf, so that the first such bit names the stage
 *   where they appeared.  A debugging aid: it reads those buffers once more
 *   (a few extra launches).  Requires d_status (null: GDN_EINVAL).  Decode
 *   ignores it. */
#define GDN_CHECK_FINITE 0x2
/* GDN_TEST_WAIT_TIMEOUT (test only): exercises the bounded waits of the
 *   tensor-core prefill.  Every wait between CTAs and warps, bounded in global
 *   time (%globaltimer) at 4 s otherwise, gives up after 2 ms, and the prep
 *   kernel does not publish the last chunk of sequence 0 for key head 0, so
 *   the scan CTAs of value heads 0 and 1 of sequence 0 time out waiting for
 *   it: they set GDN_DEV_WAIT_TIMEOUT, skip their remaining work (those
 *   heads' outputs and final states are not valid), free their tensor memory
 *   and return; the GPU context stays usable.  It takes effect only where the
 *   scan runs beside the prep (at most half as many (sequence, value head)
 *   chains as SMs); elsewhere it is ignored, as it is by the SIMT path. */
#define GDN_TEST_WAIT_TIMEOUT 0x4
/* GDN_BF16_OPERANDS: the tensor-core prefill feeds its MMAs bf16 operands
 *   (8-bit mantissa, the range of fp32) instead of fp16: the bf16 state option
 *   for precision comparisons, at the same speed.  On ordinary inputs it meets
 *   the bf16 I/O tolerance; on long runs of fully correlated keys with beta
 *   near 1 and no decay its rounding leaves several times the fp16 operands'
 *   error in the state and can take the outputs past that tolerance (the
 *   precision tests measure it).  Ignored where the SIMT path runs
 *   (GDN_FP32_STATE or other shapes). */
#define GDN_BF16_OPERANDS 0x8

typedef struct {
  int32_t h_k;     /* key/query heads */
  int32_t h_v;     /* value heads; multiple of h_k */
  int32_t d_k;     /* key head dim: 16, 32, 64 or 128 */
  int32_t d_v;     /* value head dim: 16, 32, 64 or 128 */
  int32_t conv_w;  /* conv width; must be 4 */
  int32_t chunk;   /* prefill chunk length: 16, 32, 64 or 128 (the tensor-core
                      path runs chunk 64; other lengths take the SIMT path) */
  int32_t io;      /* gdn_dtype of x, a, b, o and the conv pool */
  float l2_eps;    /* added to the sum of squares inside the L2-norm root */
  int32_t flags;   /* GDN_FP32_STATE | GDN_CHECK_FINITE | GDN_TEST_WAIT_TIMEOUT |
                      GDN_BF16_OPERANDS, or 0; other bits: GDN_EINVAL */
} gdn_dims;

typedef struct {
  const float* conv_weight; /* [conv_dim][conv_w] */
  const float* A_log;       /* [h_v] */
  const float* dt_bias;     /* [h_v] */
} gdn_params;

/*
 * gdn_conv1d_update -- one decode token per row through the causal conv:
 *   y[n][c] = SiLU( sum_w conv_weight[c][w] * hist_w[c] ),
 * hist = (conv_pool[slot][0..W-2][c], x[n][c]); then the slot's window is
 * rolled to (rows 1..W-2, x[n]).  (Vallmo README, "What's here": causal
 * conv1d; oxydllm notes, New Features, "Gated DeltaNet runtime".)
 *   x          [n][conv_dim] IO (device)
 *   conv_pool  [num_slots][W-1][conv_dim] IO (device), updated in place
 *   slot_idx   [n] int32 (device); < 0 marks a padding row (y zeroed, no
 *              window touched); >= num_slots sets GDN_DEV_BAD_SLOT
 *   y          [n][conv_dim] IO (device), post-SiLU
 * Slots must be distinct within a call.
 */
int gdn_conv1d_update(const gdn_dims* dims, const float* conv_weight,
                      const void* x, void* conv_pool, int64_t num_slots,
                      const int32_t* slot_idx, int32_t n, void* y,
                      int32_t* d_status, gdn_stream_t stream);

/*
 * gdn_gated_rmsnorm -- the DeltaNet "gated norm" on the layer output, for
 * every row of d_v values (one token, one value head):
 *   y[r][j] = o[r][j] / sqrt(mean_j o[r][j]^2 + eps) * weight[j] * SiLU(z[r][j])
 * The weight is applied as stored: of the model's norms only this one has no
 * pre-added +1 (oxydllm notes, New Features, "GGUF qwen35 architecture"); it
 * runs once over the whole token batch after the layer ("Gated DeltaNet fast
 * paths").  Used after gdn_prefill and after gdn_decode_step alike.
 *   weight     [d_v] fp32 (device)
 *   o, z       [n][h_v][d_v] IO (device)
 *   y          [n][h_v][d_v] IO (device); may be o itself (in place)
 * Uses dims->h_v, d_v (16, 32, 64 or 128) and io.  Returns GDN_EINVAL (null
 * pointer, n < 0, eps < 0), GDN_EUNSUPPORTED (d_v) or GDN_EALIGN (a pointer
 * not 16-byte aligned) without launching anything.  The caller owns every
 * buffer.
 */
int gdn_gated_rmsnorm(const gdn_dims* dims, const float* weight, float eps, const void* o,
                      const void* z, int64_t n, void* y, gdn_stream_t stream);

/*
 * gdn_gate_projection -- the decay and beta input projections of the layer
 * as one matmul over the whole token batch (oxydllm 0.0.0-alpha.12.2 release
 * notes, Performance, "Gated DeltaNet fast paths": the small beta/decay
 * projections fuse into one matmul when dense).  With W = w_ba, its rows
 * 0 .. h_v - 1 the decay projection and rows h_v .. 2 h_v - 1 the beta
 * projection:
 *   a[t][h] = sum_i hidden[t][i] W[h][i],   b[t][h] = sum_i hidden[t][i] W[h_v + h][i]
 * for t < n and h < h_v: the gate inputs a and b that gdn_prefill and
 * gdn_decode_step take.  fp32 accumulation on the tensor cores, rounded once
 * to bf16.
 *   hidden     [n][d_model] bf16 (device), the layer's input hidden states
 *   w_ba       [2 h_v][d_model] bf16 (device)
 *   a, b       [n][h_v] bf16 (device), written
 *   d_status   optional device int32: GDN_DEV_WAIT_TIMEOUT if an internal
 *              wait ran out (the outputs are then not valid)
 * Uses dims->h_v only (the inputs and outputs are bf16 whatever dims->io).
 * Returns GDN_EINVAL (null dims or pointer, n < 0, d_model <= 0, h_v <= 0),
 * GDN_EUNSUPPORTED (h_v not a multiple of 16 or above 128, d_model not a
 * multiple of 64, n above 2^31 - 1) or GDN_EALIGN (a pointer not 16-byte aligned) without
 * launching anything; n = 0 does nothing.  The caller owns every buffer.
 */
int gdn_gate_projection(const gdn_dims* dims, const void* hidden, const void* w_ba,
                        int32_t d_model, int64_t n, void* a, void* b, int32_t* d_status,
                        gdn_stream_t stream);

/* Bytes of device workspace gdn_prefill needs for this shape (0 on bad dims).
 * Library plumbing, not an operation of the method: the workspace holds the
 * per-chunk records between the state-independent stage and the scan. */
size_t gdn_prefill_workspace_size(const gdn_dims* dims, int64_t total_tokens,
                                  int32_t num_seqs);

/*
 * gdn_prefill -- the whole layer over a varlen batch, chunked (chunk length
 * dims->chunk) as the oxydllm notes describe: a chunked parallel scan for
 * prefill with the state-independent work batched ahead of the cross-chunk
 * loop (New Features, "Gated DeltaNet runtime"; Performance, "Gated DeltaNet
 * fast paths").  Each chunk's unit-lower-triangular system
 * (I + strict_tril(diag(beta) K K^T * exp(gamma_r - gamma_s)))^-1 is solved
 * by exact substitution, which stays finite on fully correlated keys.
 *   x [total_tokens][conv_dim], a, b [total_tokens][h_v] IO (device)
 *   cu_seqlens [num_seqs+1] int32 (device): 0 = cu[0] <= cu[1] <= ... =
 *              total_tokens, else GDN_DEV_BAD_CU_SEQLENS and nothing runs
 *   slot_idx [num_seqs] int32 (device), distinct; out of range (< 0 or
 *              >= num_slots) -> GDN_DEV_BAD_SLOT and that sequence is
 *              skipped: its o rows, state and window are left as they were
 *              (prefill has no padding sequences)
 *   has_initial_state [num_seqs] uint8 (device) or NULL (= all zero): when
 *              zero the sequence starts from S = 0 and an all-zero window,
 *              ignoring what its slot holds
 *   state_pool, conv_pool: read (initial state) and overwritten with the
 *              final state / last W-1 raw inputs at each sequence's slot; a
 *              zero-length sequence writes its initial (or zero) state back
 *   o [total_tokens][h_v][d_v] IO (device)
 *   workspace: device scratch of gdn_prefill_workspace_size() bytes, 256-byte
 *              aligned, owned by the caller, clobbered by the call.
 */
int gdn_prefill(const gdn_dims* dims, const gdn_params* params,
                const void* x, const void* a, const void* b,
                const int32_t* cu_seqlens, int32_t num_seqs,
                int64_t total_tokens, const int32_t* slot_idx,
                const uint8_t* has_initial_state, float* state_pool,
                void* conv_pool, int64_t num_slots, void* o,
                void* workspace, size_t workspace_bytes, int32_t* d_status,
                gdn_stream_t stream);

/*
 * gdn_decode_step -- one token for each of n rows, O(1) in sequence length
 * (oxydllm notes, New Features, "Gated DeltaNet runtime": the recurrent step
 * for decode).  Row n uses slot s = slot_idx[n]: the conv runs on the slot's
 * window plus x[n] and rolls the window, then the slot's state is read once
 * and written once:
 *   u = S k^, r = S q^, delta = beta (v - alpha u),
 *   S' = alpha S + delta k^T, o = alpha r + delta (k^ . q^),  alpha = e^g,
 * which equals the recurrence above for one token.
 *   x [n][conv_dim], a, b [n][h_v] IO (device); slot_idx [n] int32 (device),
 *   distinct, < 0 = padding row (o zeroed, nothing else touched);
 *   o [n][h_v][d_v] IO (device).
 */
int gdn_decode_step(const gdn_dims* dims, const gdn_params* params,
                    const void* x, const void* a, const void* b,
                    const int32_t* slot_idx, int32_t n, float* state_pool,
                    void* conv_pool, int64_t num_slots, void* o,
                    int32_t* d_status, gdn_stream_t stream);

/*
 * Stage tracing for gdn_prefill_traced.  Each non-NULL handle is a CUDA event
 * (cudaEvent_t) owned by the caller; the call records begin[i] on `stream`
 * right before stage i's first kernel and end[i] right after its last kernel,
 * sets `launches` to the number of kernels the call enqueued and `stages_run`
 * to a bit mask of the stages it ran.  A stage the call does not run records
 * nothing.
 *   stage 0  front end: argument check on the device, conv + SiLU, L2 norm,
 *            gates, conv-window write-back
 *   stage 1  per-chunk state-independent work (on the tensor-core path it
 *            is part of stage 2 when the prep and the scan run overlapped)
 *   stage 2  cross-chunk state scan and outputs
 */
#define GDN_NUM_STAGES 3
typedef struct {
  void* begin[GDN_NUM_STAGES];
  void* end[GDN_NUM_STAGES];
  int32_t launches;   /* written by the call */
  int32_t stages_run; /* written by the call: bit i = stage i ran */
} gdn_trace;

/* gdn_prefill with stage tracing; trace may be NULL (then identical to
 * gdn_prefill).  Instrumentation for measuring the stages, not an operation
 * of the method. */
int gdn_prefill_traced(const gdn_dims* dims, const gdn_params* params,
                       const void* x, const void* a, const void* b,
                       const int32_t* cu_seqlens, int32_t num_seqs,
                       int64_t total_tokens, const int32_t* slot_idx,
                       const uint8_t* has_initial_state, float* state_pool,
                       void* conv_pool, int64_t num_slots, void* o,
                       void* workspace, size_t workspace_bytes,
                       int32_t* d_status, gdn_trace* trace,
                       gdn_stream_t stream);

/*
 * gdn_prefill_noalloc -- gdn_prefill for callers that cannot allocate device
 * memory (a deployment variant; the pages define no such call).  Code
 * running inside a host framework whose allocator already owns nearly all of
 * HBM, or on a path where cudaMalloc's implicit synchronisation is not
 * acceptable, cannot obtain the workspace gdn_prefill wants.  This entry point
 * takes the same arguments minus the workspace and uses a scratch array of
 * GDN_NOALLOC_SCRATCH_BYTES that is part of the library's device image: every
 * GPU that loads the library holds those bytes until the process exits.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Returns GDN_EWORKSPACE, with nothing enqueued, when the call would need
 *     more than GDN_NOALLOC_SCRATCH_BYTES of workspace.  The rule is
 *     gdn_prefill_workspace_size(dims, total_tokens, num_seqs) <=
 *     GDN_NOALLOC_SCRATCH_BYTES; at the Qwen3.5-4B layer shape that is about
 *     1.87 MB per chunk slot on the tensor-core path (ceil(len / 64) slots per
 *     sequence, so 2176 tokens for one sequence, fewer as sequences are added)
 *     and about 74 KB per token with GDN_FP32_STATE (896 tokens).
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for the
 *     life of the process; make that first call before any stream capture.
 *     The device must not be reset (cudaDeviceReset, or any teardown of its
 *     primary context) while the library is loaded: the array may then live
 *     at another address and the cached one would be stale.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (nothing in it needs to start at zero).  Calls whose
 *     kernels overlap on the GPU (different streams, or different host
 *     threads) race on it: serialise them.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
int gdn_prefill_noalloc(const gdn_dims* dims, const gdn_params* params,
                        const void* x, const void* a, const void* b,
                        const int32_t* cu_seqlens, int32_t num_seqs,
                        int64_t total_tokens, const int32_t* slot_idx,
                        const uint8_t* has_initial_state, float* state_pool,
                        void* conv_pool, int64_t num_slots, void* o,
                        int32_t* d_status, gdn_stream_t stream);

/*
 * gdn_prefill_checkpointed -- gdn_prefill that also leaves interval
 * checkpoints of each sequence's recurrent state in other slots of the same
 * pools (PicoLM changelog, "SSM State Checkpointing": checkpoints every N
 * tokens during prefill; on a partial prefix match the closest checkpoint is
 * restored and only the remaining tokens are processed).  Same arguments as
 * gdn_prefill plus:
 *   ckpt_every  interval in tokens: a positive multiple of dims->chunk, else
 *               GDN_EINVAL with nothing enqueued
 *   ckpt_slot   device int32 [num_seqs]: first checkpoint slot of each
 *               sequence; < 0 = no checkpoints for it.  NULL: GDN_EINVAL.
 * For sequence b and every k >= 1 with k * ckpt_every < len_b, slot
 * ckpt_slot[b] + k - 1 receives the state (fp32 [h_v][d_k][d_v], S^T) and the
 * conv window (the last conv_w - 1 raw inputs) after the first k * ckpt_every
 * tokens of the sequence, its initial state and window included -- exactly
 * what a gdn_prefill of that prefix would leave in its slot, so a prefill of
 * the remaining tokens from that slot (has_initial_state = 1) continues the
 * sequence.  The final state goes to slot_idx[b] as in gdn_prefill.  A
 * checkpoint slot >= num_slots sets GDN_DEV_BAD_SLOT in *d_status and that
 * checkpoint is skipped.  Checkpoint slots must differ from every slot the
 * call reads or writes otherwise (the caller's contract; overlaps are
 * undefined).  Costs one extra state write per checkpoint.
 */
int gdn_prefill_checkpointed(const gdn_dims* dims, const gdn_params* params,
                             const void* x, const void* a, const void* b,
                             const int32_t* cu_seqlens, int32_t num_seqs,
                             int64_t total_tokens, const int32_t* slot_idx,
                             const uint8_t* has_initial_state, float* state_pool,
                             void* conv_pool, int64_t num_slots, void* o,
                             void* workspace, size_t workspace_bytes,
                             int64_t ckpt_every, const int32_t* ckpt_slot,
                             int32_t* d_status, gdn_stream_t stream);

/*
 * gdn_slot_copy -- copy whole recurrent slots: for each i < n, slot
 * dst_slot[i] receives the state and conv window of slot src_slot[i].
 * Snapshot (a live slot to a spare one), restore (back) and fork (one prefix
 * into several sequences) are this copy (Vallmo.jl README, src/: recurrent
 * state snapshotted and restored for prefix caching; PicoLM changelog, "SSM
 * State Checkpointing": capture and restore the full SSM state).
 *   state_pool  device fp32 [num_slots][h_v][d_k][d_v], 16-byte aligned
 *   conv_pool   device I/O dtype [num_slots][conv_w-1][conv_dim], 16-byte aligned
 *   src_slot, dst_slot  device int32 [n]; a pair with either < 0 is padding and
 *               skipped; src == dst is a no-op; either >= num_slots sets
 *               GDN_DEV_BAD_SLOT in *d_status and that pair is skipped
 * Host-checkable problems (bad dims, NULL pointers with n > 0, misalignment,
 * n < 0) return an error with nothing enqueued.  The pairs are copied
 * concurrently: a slot that is one pair's destination must not be another
 * pair's source or destination (undefined otherwise).  HBM-bound: each pair
 * reads and writes the state and window bytes once.
 */
int gdn_slot_copy(const gdn_dims* dims, float* state_pool, void* conv_pool,
                  int64_t num_slots, const int32_t* src_slot, const int32_t* dst_slot,
                  int32_t n, int32_t* d_status, gdn_stream_t stream);

/*
 * gdn_prefill_gated_norm / gdn_decode_step_gated_norm -- gdn_prefill and
 * gdn_decode_step followed by the gated RMSNorm of the layer output (the norm
 * that follows the Gated DeltaNet core in the Qwen3.5 layer: oxydllm release
 * notes, New Features, GGUF qwen35 architecture and "Gated DeltaNet fast
 * paths"; PicoLM changelog, SSM/GDN kernel notes): instead of o they write
 *     y[t][h][:] = o[t][h][:] / sqrt(mean_j o[t][h][j]^2 + eps) * w * SiLU(z[t][h][:])
 * exactly as gdn_gated_rmsnorm defines it.  Same arguments as gdn_prefill /
 * gdn_decode_step, with the output o replaced by:
 *   z            device, I/O dtype, [total_tokens or n][h_v][d_v], 16-byte aligned
 *   norm_weight  device fp32 [d_v], 16-byte aligned
 *   eps          >= 0 (NaN or negative: GDN_EINVAL)
 *   y            device, I/O dtype, [total_tokens or n][h_v][d_v]; must not
 *                overlap z (y == z: GDN_EINVAL) nor any other input
 * In decode the norm runs in the step's own epilogue (one CTA holds a head's
 * whole output row), so o never reaches memory.  In prefill the layer writes o
 * into y and the standalone norm kernel rewrites it in place on the same
 * stream: the scans spread a token's values over several warps (tensor-core
 * path) or CTAs (SIMT path), and a norm inside the tensor-core scan's output
 * warps lengthened its chunk period, so two launches are the faster order.
 */
int gdn_prefill_gated_norm(const gdn_dims* dims, const gdn_params* params,
                           const void* x, const void* a, const void* b,
                           const int32_t* cu_seqlens, int32_t num_seqs,
                           int64_t total_tokens, const int32_t* slot_idx,
                           const uint8_t* has_initial_state, float* state_pool,
                           void* conv_pool, int64_t num_slots, const void* z,
                           const float* norm_weight, float eps, void* y,
                           void* workspace, size_t workspace_bytes,
                           int32_t* d_status, gdn_stream_t stream);
int gdn_decode_step_gated_norm(const gdn_dims* dims, const gdn_params* params,
                               const void* x, const void* a, const void* b,
                               const int32_t* slot_idx, int32_t n, float* state_pool,
                               void* conv_pool, int64_t num_slots, const void* z,
                               const float* norm_weight, float eps, void* y,
                               int32_t* d_status, gdn_stream_t stream);

/* Static description of a gdn_status code (library plumbing).  The string is
 * owned by the library and valid for the life of the process. */
const char* gdn_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
