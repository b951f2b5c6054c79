"""Thin ctypes binding of libgdn_gb300.so (include/gdn.h), same names as the C
ABI.  It only marshals arguments: shapes and device pointers of torch tensors
go in, a non-zero gdn_status comes back as GdnError.  Every step of the layer
runs in the library's CUDA kernels; there is no Python or CPU fallback, and
loading fails loudly when the library has not been built."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgdn_gb300.so")

GDN_FP32, GDN_BF16 = 0, 1
GDN_DEV_BAD_SLOT, GDN_DEV_BAD_CU_SEQLENS, GDN_DEV_WAIT_TIMEOUT = 0x1, 0x2, 0x4
GDN_FP32_STATE = 0x1   # gdn_dims.flags: fp32 state products in prefill
GDN_CHECK_FINITE = 0x2  # gdn_dims.flags: per-stage NaN/Inf probe of prefill
GDN_TEST_WAIT_TIMEOUT = 0x4  # gdn_dims.flags (tests only): 2 ms waits, one chunk withheld
GDN_BF16_OPERANDS = 0x8      # gdn_dims.flags: bf16 instead of fp16 tensor-core operands
GDN_DEV_NONFINITE_FRONTEND, GDN_DEV_NONFINITE_CHUNK, GDN_DEV_NONFINITE_OUT = 0x8, 0x10, 0x20
STATUS = {0: "GDN_OK", -1: "GDN_EINVAL", -2: "GDN_EUNSUPPORTED", -3: "GDN_ECUDA",
          -4: "GDN_EWORKSPACE", -5: "GDN_EALIGN"}

_lib = None


class GdnError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        msg = _lib.gdn_status_str(status).decode() if _lib is not None else ""
        super().__init__(f"{func} returned {STATUS.get(status, status)} ({msg})")


class gdn_dims(ctypes.Structure):
    _fields_ = [("h_k", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("conv_w", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("io", ctypes.c_int32), ("l2_eps", ctypes.c_float), ("flags", ctypes.c_int32)]


class gdn_params(ctypes.Structure):
    _fields_ = [("conv_weight", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p)]


GDN_NUM_STAGES = 3
STAGES = ("frontend", "chunk", "scan")


class gdn_trace(ctypes.Structure):
    _fields_ = [("begin", ctypes.c_void_p * GDN_NUM_STAGES),
                ("end", ctypes.c_void_p * GDN_NUM_STAGES),
                ("launches", ctypes.c_int32), ("stages_run", ctypes.c_int32)]


def make_dims(h_k, h_v, d_k, d_v, chunk=64, io="bf16", conv_w=4, l2_eps=1e-6,
              flags=0) -> gdn_dims:
    io_code = {"fp32": GDN_FP32, "bf16": GDN_BF16}[io] if isinstance(io, str) else int(io)
    return gdn_dims(h_k, h_v, d_k, d_v, conv_w, chunk, io_code, l2_eps, flags)


def dims_from(d) -> gdn_dims:
    """gdn_dims from any object with h_k, h_v, d_k, d_v, chunk, io, conv_w, l2_eps
    (and optionally flags)."""
    if isinstance(d, gdn_dims):
        return d
    return make_dims(d.h_k, d.h_v, d.d_k, d.d_v, d.chunk, d.io, d.conv_w, d.l2_eps,
                     getattr(d, "flags", 0))


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D, PR = ctypes.POINTER(gdn_dims), ctypes.POINTER(gdn_params)
    lib.gdn_status_str.argtypes = [ctypes.c_int]
    lib.gdn_status_str.restype = ctypes.c_char_p
    lib.gdn_conv1d_update.argtypes = [D, P, P, P, I64, P, I32, P, P, P]
    lib.gdn_conv1d_update.restype = ctypes.c_int
    lib.gdn_prefill_workspace_size.argtypes = [D, I64, I32]
    lib.gdn_prefill_workspace_size.restype = SZ
    lib.gdn_prefill.argtypes = [D, PR, P, P, P, P, I32, I64, P, P, P, P, I64, P, P, SZ, P, P]
    lib.gdn_prefill.restype = ctypes.c_int
    lib.gdn_prefill_traced.argtypes = [D, PR, P, P, P, P, I32, I64, P, P, P, P, I64, P, P, SZ, P,
                                       ctypes.POINTER(gdn_trace), P]
    lib.gdn_prefill_traced.restype = ctypes.c_int
    lib.gdn_prefill_noalloc.argtypes = [D, PR, P, P, P, P, I32, I64, P, P, P, P, I64, P, P, P]
    lib.gdn_prefill_noalloc.restype = ctypes.c_int
    lib.gdn_decode_step.argtypes = [D, PR, P, P, P, P, I32, P, P, I64, P, P, P]
    lib.gdn_decode_step.restype = ctypes.c_int
    lib.gdn_gated_rmsnorm.argtypes = [D, P, ctypes.c_float, P, P, I64, P, P]
    lib.gdn_gated_rmsnorm.restype = ctypes.c_int
    lib.gdn_prefill_checkpointed.argtypes = [D, PR, P, P, P, P, I32, I64, P, P, P, P, I64, P, P,
                                             SZ, I64, P, P, P]
    lib.gdn_prefill_checkpointed.restype = ctypes.c_int
    lib.gdn_slot_copy.argtypes = [D, P, P, I64, P, P, I32, P, P]
    lib.gdn_slot_copy.restype = ctypes.c_int
    F = ctypes.c_float
    lib.gdn_prefill_gated_norm.argtypes = [D, PR, P, P, P, P, I32, I64, P, P, P, P, I64, P, P, F,
                                           P, P, SZ, P, P]
    lib.gdn_prefill_gated_norm.restype = ctypes.c_int
    lib.gdn_decode_step_gated_norm.argtypes = [D, PR, P, P, P, P, I32, P, P, I64, P, P, F, P, P, P]
    lib.gdn_decode_step_gated_norm.restype = ctypes.c_int
    lib.gdn_gate_projection.argtypes = [D, P, P, I32, I64, P, P, P, P]
    lib.gdn_gate_projection.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(func, rc):
    if rc != 0:
        raise GdnError(func, rc)


def _io_dtype(d: gdn_dims):
    import torch
    return torch.bfloat16 if d.io == GDN_BF16 else torch.float32


def _expect(t, name, dtype=None, numel=None):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def conv_dim(d: gdn_dims) -> int:
    return 2 * d.h_k * d.d_k + d.h_v * d.d_v


def gdn_prefill_workspace_size(dims, total_tokens: int, num_seqs: int) -> int:
    d = dims_from(dims)
    return int(load().gdn_prefill_workspace_size(ctypes.byref(d), int(total_tokens), int(num_seqs)))


def gdn_conv1d_update(dims, conv_weight, x, conv_pool, slot_idx, y, d_status=None, stream=None):
    import torch
    d = dims_from(dims)
    n = int(slot_idx.numel())
    io = _io_dtype(d)
    _expect(conv_weight, "conv_weight", torch.float32, conv_dim(d) * d.conv_w)
    _expect(x, "x", io, n * conv_dim(d))
    _expect(y, "y", io, n * conv_dim(d))
    _expect(conv_pool, "conv_pool", io)
    _expect(slot_idx, "slot_idx", torch.int32)
    num_slots = conv_pool.numel() // ((d.conv_w - 1) * conv_dim(d))
    rc = load().gdn_conv1d_update(ctypes.byref(d), _ptr(conv_weight), _ptr(x), _ptr(conv_pool),
                                  num_slots, _ptr(slot_idx), n, _ptr(y), _ptr(d_status),
                                  _stream(stream))
    _check("gdn_conv1d_update", rc)


def gdn_prefill(dims, conv_weight, A_log, dt_bias, x, a, b, cu_seqlens, slot_idx,
                has_initial_state, state_pool, conv_pool, o, workspace, d_status=None,
                stream=None, trace=None):
    """Whole layer over a varlen batch (see gdn_prefill in include/gdn.h).

    trace: optional gdn_trace (stage events + launch count); when given the call
    goes through gdn_prefill_traced."""
    import torch
    d = dims_from(dims)
    io = _io_dtype(d)
    B = int(cu_seqlens.numel()) - 1
    T = int(x.shape[0]) if x is not None else 0
    cd = conv_dim(d)
    _expect(conv_weight, "conv_weight", torch.float32, cd * d.conv_w)
    _expect(A_log, "A_log", torch.float32, d.h_v)
    _expect(dt_bias, "dt_bias", torch.float32, d.h_v)
    _expect(x, "x", io, T * cd)
    _expect(a, "a", io, T * d.h_v)
    _expect(b, "b", io, T * d.h_v)
    _expect(o, "o", io, T * d.h_v * d.d_v)
    _expect(cu_seqlens, "cu_seqlens", torch.int32)
    _expect(slot_idx, "slot_idx", torch.int32, B)
    _expect(has_initial_state, "has_initial_state", torch.uint8, B)
    _expect(state_pool, "state_pool", torch.float32)
    _expect(conv_pool, "conv_pool", io)
    num_slots = state_pool.numel() // (d.h_v * d.d_k * d.d_v)
    p = gdn_params(conv_weight.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr())
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (ctypes.byref(d), ctypes.byref(p), _ptr(x), _ptr(a), _ptr(b), _ptr(cu_seqlens), B, T,
            _ptr(slot_idx), _ptr(has_initial_state), _ptr(state_pool), _ptr(conv_pool),
            num_slots, _ptr(o), _ptr(workspace), ws_bytes, _ptr(d_status))
    if trace is None:
        _check("gdn_prefill", load().gdn_prefill(*args, _stream(stream)))
    else:
        _check("gdn_prefill_traced",
               load().gdn_prefill_traced(*args, ctypes.byref(trace), _stream(stream)))


def gdn_prefill_checkpointed(dims, conv_weight, A_log, dt_bias, x, a, b, cu_seqlens, slot_idx,
                             has_initial_state, state_pool, conv_pool, o, workspace, ckpt_every,
                             ckpt_slot, d_status=None, stream=None):
    """gdn_prefill plus interval checkpoints: every ckpt_every tokens (a multiple
    of the chunk) strictly inside sequence b, its state and conv window go to
    slot ckpt_slot[b] + k - 1 (see gdn_prefill_checkpointed in include/gdn.h)."""
    import torch
    d = dims_from(dims)
    io = _io_dtype(d)
    B = int(cu_seqlens.numel()) - 1
    T = int(x.shape[0]) if x is not None else 0
    cd = conv_dim(d)
    _expect(conv_weight, "conv_weight", torch.float32, cd * d.conv_w)
    _expect(A_log, "A_log", torch.float32, d.h_v)
    _expect(dt_bias, "dt_bias", torch.float32, d.h_v)
    _expect(x, "x", io, T * cd)
    _expect(a, "a", io, T * d.h_v)
    _expect(b, "b", io, T * d.h_v)
    _expect(o, "o", io, T * d.h_v * d.d_v)
    _expect(cu_seqlens, "cu_seqlens", torch.int32)
    _expect(slot_idx, "slot_idx", torch.int32, B)
    _expect(has_initial_state, "has_initial_state", torch.uint8, B)
    _expect(ckpt_slot, "ckpt_slot", torch.int32, B)
    _expect(state_pool, "state_pool", torch.float32)
    _expect(conv_pool, "conv_pool", io)
    num_slots = state_pool.numel() // (d.h_v * d.d_k * d.d_v)
    p = gdn_params(conv_weight.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr())
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("gdn_prefill_checkpointed", load().gdn_prefill_checkpointed(
        ctypes.byref(d), ctypes.byref(p), _ptr(x), _ptr(a), _ptr(b), _ptr(cu_seqlens), B, T,
        _ptr(slot_idx), _ptr(has_initial_state), _ptr(state_pool), _ptr(conv_pool), num_slots,
        _ptr(o), _ptr(workspace), ws_bytes, int(ckpt_every), _ptr(ckpt_slot), _ptr(d_status),
        _stream(stream)))


def gdn_prefill_gated_norm(dims, conv_weight, A_log, dt_bias, x, a, b, cu_seqlens, slot_idx,
                           has_initial_state, state_pool, conv_pool, z, norm_weight, y, workspace,
                           eps=1e-6, d_status=None, stream=None):
    """gdn_prefill with the gated RMSNorm of the output fused in: writes
    y = rmsnorm(o) * norm_weight * SiLU(z) (see gdn_prefill_gated_norm in
    include/gdn.h)."""
    import torch
    d = dims_from(dims)
    io = _io_dtype(d)
    B = int(cu_seqlens.numel()) - 1
    T = int(x.shape[0]) if x is not None else 0
    cd = conv_dim(d)
    _expect(conv_weight, "conv_weight", torch.float32, cd * d.conv_w)
    _expect(A_log, "A_log", torch.float32, d.h_v)
    _expect(dt_bias, "dt_bias", torch.float32, d.h_v)
    _expect(x, "x", io, T * cd)
    _expect(a, "a", io, T * d.h_v)
    _expect(b, "b", io, T * d.h_v)
    _expect(z, "z", io, T * d.h_v * d.d_v)
    _expect(y, "y", io, T * d.h_v * d.d_v)
    _expect(norm_weight, "norm_weight", torch.float32, d.d_v)
    _expect(cu_seqlens, "cu_seqlens", torch.int32)
    _expect(slot_idx, "slot_idx", torch.int32, B)
    _expect(has_initial_state, "has_initial_state", torch.uint8, B)
    _expect(state_pool, "state_pool", torch.float32)
    _expect(conv_pool, "conv_pool", io)
    num_slots = state_pool.numel() // (d.h_v * d.d_k * d.d_v)
    p = gdn_params(conv_weight.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr())
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("gdn_prefill_gated_norm", load().gdn_prefill_gated_norm(
        ctypes.byref(d), ctypes.byref(p), _ptr(x), _ptr(a), _ptr(b), _ptr(cu_seqlens), B, T,
        _ptr(slot_idx), _ptr(has_initial_state), _ptr(state_pool), _ptr(conv_pool), num_slots,
        _ptr(z), _ptr(norm_weight), float(eps), _ptr(y), _ptr(workspace), ws_bytes,
        _ptr(d_status), _stream(stream)))


def gdn_decode_step_gated_norm(dims, conv_weight, A_log, dt_bias, x, a, b, slot_idx, state_pool,
                               conv_pool, z, norm_weight, y, eps=1e-6, d_status=None, stream=None):
    """gdn_decode_step with the gated RMSNorm of the output fused in (see
    gdn_decode_step_gated_norm in include/gdn.h)."""
    import torch
    d = dims_from(dims)
    io = _io_dtype(d)
    n = int(slot_idx.numel())
    cd = conv_dim(d)
    _expect(conv_weight, "conv_weight", torch.float32, cd * d.conv_w)
    _expect(A_log, "A_log", torch.float32, d.h_v)
    _expect(dt_bias, "dt_bias", torch.float32, d.h_v)
    _expect(x, "x", io, n * cd)
    _expect(a, "a", io, n * d.h_v)
    _expect(b, "b", io, n * d.h_v)
    _expect(z, "z", io, n * d.h_v * d.d_v)
    _expect(y, "y", io, n * d.h_v * d.d_v)
    _expect(norm_weight, "norm_weight", torch.float32, d.d_v)
    _expect(slot_idx, "slot_idx", torch.int32, n)
    _expect(state_pool, "state_pool", torch.float32)
    _expect(conv_pool, "conv_pool", io)
    num_slots = state_pool.numel() // (d.h_v * d.d_k * d.d_v)
    p = gdn_params(conv_weight.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr())
    _check("gdn_decode_step_gated_norm", load().gdn_decode_step_gated_norm(
        ctypes.byref(d), ctypes.byref(p), _ptr(x), _ptr(a), _ptr(b), _ptr(slot_idx), n,
        _ptr(state_pool), _ptr(conv_pool), num_slots, _ptr(z), _ptr(norm_weight), float(eps),
        _ptr(y), _ptr(d_status), _stream(stream)))


def gdn_slot_copy(dims, state_pool, conv_pool, src_slot, dst_slot, d_status=None, stream=None):
    """Copy whole slots (state and conv window): slot dst_slot[i] <- slot
    src_slot[i]; padding pairs (< 0) skipped (see gdn_slot_copy in include/gdn.h)."""
    import torch
    d = dims_from(dims)
    _expect(state_pool, "state_pool", torch.float32)
    _expect(conv_pool, "conv_pool", _io_dtype(d))
    n = int(src_slot.numel())
    _expect(src_slot, "src_slot", torch.int32, n)
    _expect(dst_slot, "dst_slot", torch.int32, n)
    num_slots = state_pool.numel() // (d.h_v * d.d_k * d.d_v)
    _check("gdn_slot_copy", load().gdn_slot_copy(
        ctypes.byref(d), _ptr(state_pool), _ptr(conv_pool), num_slots, _ptr(src_slot),
        _ptr(dst_slot), n, _ptr(d_status), _stream(stream)))


GDN_NOALLOC_SCRATCH_BYTES = 64 << 20


def gdn_prefill_noalloc(dims, conv_weight, A_log, dt_bias, x, a, b, cu_seqlens, slot_idx,
                        has_initial_state, state_pool, conv_pool, o, d_status=None, stream=None):
    """gdn_prefill without a workspace argument, for callers that cannot allocate
    device memory: the library uses its own fixed device scratch array of
    GDN_NOALLOC_SCRATCH_BYTES (see gdn_prefill_noalloc in include/gdn.h)."""
    import torch
    d = dims_from(dims)
    io = _io_dtype(d)
    B = int(cu_seqlens.numel()) - 1
    T = int(x.shape[0]) if x is not None else 0
    cd = conv_dim(d)
    _expect(conv_weight, "conv_weight", torch.float32, cd * d.conv_w)
    _expect(A_log, "A_log", torch.float32, d.h_v)
    _expect(dt_bias, "dt_bias", torch.float32, d.h_v)
    _expect(x, "x", io, T * cd)
    _expect(a, "a", io, T * d.h_v)
    _expect(b, "b", io, T * d.h_v)
    _expect(o, "o", io, T * d.h_v * d.d_v)
    _expect(cu_seqlens, "cu_seqlens", torch.int32)
    _expect(slot_idx, "slot_idx", torch.int32, B)
    _expect(has_initial_state, "has_initial_state", torch.uint8, B)
    _expect(state_pool, "state_pool", torch.float32)
    _expect(conv_pool, "conv_pool", io)
    num_slots = state_pool.numel() // (d.h_v * d.d_k * d.d_v)
    p = gdn_params(conv_weight.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr())
    rc = load().gdn_prefill_noalloc(ctypes.byref(d), ctypes.byref(p), _ptr(x), _ptr(a), _ptr(b),
                                    _ptr(cu_seqlens), B, T, _ptr(slot_idx),
                                    _ptr(has_initial_state), _ptr(state_pool), _ptr(conv_pool),
                                    num_slots, _ptr(o), _ptr(d_status), _stream(stream))
    _check("gdn_prefill_noalloc", rc)


def make_trace(begin_events=None, end_events=None) -> gdn_trace:
    """gdn_trace from lists (per stage) of torch.cuda.Event or None."""
    tr = gdn_trace()
    for i in range(GDN_NUM_STAGES):
        for dst, evs in ((tr.begin, begin_events), (tr.end, end_events)):
            ev = evs[i] if evs is not None else None
            dst[i] = ev.cuda_event if ev is not None else None
    return tr


def gdn_decode_step(dims, conv_weight, A_log, dt_bias, x, a, b, slot_idx, state_pool,
                    conv_pool, o, d_status=None, stream=None):
    """One decode token per row (see gdn_decode_step in include/gdn.h)."""
    import torch
    d = dims_from(dims)
    io = _io_dtype(d)
    n = int(slot_idx.numel())
    cd = conv_dim(d)
    _expect(conv_weight, "conv_weight", torch.float32, cd * d.conv_w)
    _expect(A_log, "A_log", torch.float32, d.h_v)
    _expect(dt_bias, "dt_bias", torch.float32, d.h_v)
    _expect(x, "x", io, n * cd)
    _expect(a, "a", io, n * d.h_v)
    _expect(b, "b", io, n * d.h_v)
    _expect(o, "o", io, n * d.h_v * d.d_v)
    _expect(slot_idx, "slot_idx", torch.int32)
    _expect(state_pool, "state_pool", torch.float32)
    _expect(conv_pool, "conv_pool", io)
    num_slots = state_pool.numel() // (d.h_v * d.d_k * d.d_v)
    p = gdn_params(conv_weight.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr())
    rc = load().gdn_decode_step(ctypes.byref(d), ctypes.byref(p), _ptr(x), _ptr(a), _ptr(b),
                                _ptr(slot_idx), n, _ptr(state_pool), _ptr(conv_pool), num_slots,
                                _ptr(o), _ptr(d_status), _stream(stream))
    _check("gdn_decode_step", rc)


def gdn_gated_rmsnorm(dims, weight, o, z, y=None, eps=1e-6, stream=None):
    """Gated RMSNorm of the layer output (see gdn_gated_rmsnorm in
    include/gdn.h): o, z [n, h_v, d_v] in the I/O dtype, weight [d_v] fp32;
    y defaults to o (in place).  Returns y."""
    import torch
    d = dims_from(dims)
    io = _io_dtype(d)
    n = int(o.numel()) // (d.h_v * d.d_v) if d.h_v * d.d_v else 0
    y = o if y is None else y
    _expect(weight, "weight", torch.float32, d.d_v)
    _expect(o, "o", io, n * d.h_v * d.d_v)
    _expect(z, "z", io, n * d.h_v * d.d_v)
    _expect(y, "y", io, n * d.h_v * d.d_v)
    rc = load().gdn_gated_rmsnorm(ctypes.byref(d), _ptr(weight), float(eps), _ptr(o), _ptr(z), n,
                                  _ptr(y), _stream(stream))
    _check("gdn_gated_rmsnorm", rc)
    return y


def gdn_gate_projection(dims, hidden, w_ba, a=None, b=None, d_status=None, stream=None):
    """The decay and beta input projections as one matmul (see
    gdn_gate_projection in include/gdn.h): hidden [n, d_model] bf16, w_ba
    [2 h_v, d_model] bf16 (decay rows, then beta rows) -> a, b [n, h_v] bf16
    (allocated when not given).  Returns (a, b)."""
    import torch
    d = dims_from(dims)
    if hidden.dim() != 2:
        raise ValueError("hidden must be [n, d_model]")
    n, d_model = int(hidden.shape[0]), int(hidden.shape[1])
    if a is None:
        a = torch.empty((n, d.h_v), dtype=torch.bfloat16, device=hidden.device)
    if b is None:
        b = torch.empty((n, d.h_v), dtype=torch.bfloat16, device=hidden.device)
    _expect(hidden, "hidden", torch.bfloat16)
    _expect(w_ba, "w_ba", torch.bfloat16, 2 * d.h_v * d_model)
    _expect(a, "a", torch.bfloat16, n * d.h_v)
    _expect(b, "b", torch.bfloat16, n * d.h_v)
    _expect(d_status, "d_status", torch.int32, 1)
    rc = load().gdn_gate_projection(ctypes.byref(d), _ptr(hidden), _ptr(w_ba), d_model, n,
                                    _ptr(a), _ptr(b), _ptr(d_status), _stream(stream))
    _check("gdn_gate_projection", rc)
    return a, b
