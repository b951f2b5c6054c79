"""Gated DeltaNet linear-attention layer for GB300 (sm_103a): C-ABI CUDA library
and its thin Python binding."""
