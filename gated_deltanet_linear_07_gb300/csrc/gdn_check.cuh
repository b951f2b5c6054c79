// gdn_check.cuh -- the NaN/Inf probe behind GDN_CHECK_FINITE (a debugging aid
// in the spirit of the per-stage NaN/Inf check of the oxydllm release notes,
// Performance, "Gated DeltaNet fast paths", OXYDLLM_GDN_DEBUG).  After a
// prefill call each launch below scans what one stage of the call wrote and
// ORs that stage's GDN_DEV_NONFINITE_* bit into the device status word.  Only
// rows of sequences whose slot is in range are scanned (the others are not
// written); nothing runs when cu_seqlens was rejected.
#pragma once
#include "gdn_common.cuh"

// Token-major rows: row t < total_tokens holds row_elems values (fp32, or bf16
// when bf16 is set) at p + t * row_elems.
cudaError_t gdn_check_rows(const GdnPrefillArgs& a, const void* p, bool bf16, int64_t row_elems,
                           int bit, cudaStream_t s);
// The final state of every (sequence with a valid slot, value head).
cudaError_t gdn_check_states(const GdnPrefillArgs& a, int d_k, int d_v, int bit, cudaStream_t s);
// The tensor-core path's chunk records: the [Q; K] tiles (the front end's
// output) and the value-head records P, U^T, decay factors, Wk (the chunk
// stage's output), for every chunk of a sequence with a valid slot.
cudaError_t gdn_check_tc_records(const GdnPrefillArgs& a, cudaStream_t s);
