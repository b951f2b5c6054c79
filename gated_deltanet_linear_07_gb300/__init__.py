"""Gated DeltaNet linear-attention layer for GB300 (sm_103a).

The compute lives in libgdn_gb300.so, a C-ABI CUDA library (include/gdn.h);
this package is its thin ctypes binding (same function names), the in-tree
build step and the seeded synthetic workloads.  There is no CPU or Python
fallback for any step of the layer.
"""
from ._binding import (GDN_BF16, GDN_DEV_BAD_CU_SEQLENS, GDN_DEV_BAD_SLOT,  # noqa: F401
                       GDN_DEV_WAIT_TIMEOUT, GDN_FP32, GDN_FP32_STATE, GDN_CHECK_FINITE,
                       GDN_TEST_WAIT_TIMEOUT, GDN_BF16_OPERANDS,
                       GDN_DEV_NONFINITE_FRONTEND, GDN_DEV_NONFINITE_CHUNK, GDN_DEV_NONFINITE_OUT,
                       GdnError, conv_dim, dims_from,
                       gdn_conv1d_update, gdn_decode_step, gdn_dims, gdn_gated_rmsnorm, gdn_params,
                       gdn_prefill_checkpointed, gdn_slot_copy, gdn_prefill_gated_norm,
                       gdn_decode_step_gated_norm, gdn_gate_projection,
                       gdn_prefill, gdn_prefill_noalloc, gdn_prefill_workspace_size,
                       GDN_NOALLOC_SCRATCH_BYTES, gdn_trace, load, make_dims,
                       make_trace, STAGES)
from ._build import build  # noqa: F401
