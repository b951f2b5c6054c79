"""float64 CPU oracle of the Gated DeltaNet layer (ctypes wrapper over gdn_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the package entry point's smoke check
and the benchmark's CPU-baseline leg may use it; the CUDA library and its Python
binding never import it.  The C code follows the method token by token in
float64 (see gdn_oracle.h for the statement of what it computes and which page
each step comes from).

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: brute-force evaluation of the unrolled recurrence, an
independent chunked (WY) evaluation, closed forms (pure decay, exact recall,
repeated-key overwrite), library routines for the conv/SiLU/softplus/sigmoid
front end, a hand-worked example and channel selection for the decay/beta
projection, and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lib = None

L2_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into a shared library next to it (plain gcc, -O2,
    strict IEEE double: no fast-math, no host-specific tuning)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "gdn_oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, dbl, p = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.oracle_gdn_recurrence.argtypes = [i64, i64, i64, p, p, p, p, p, p, p, p]
    lib.oracle_gdn_recurrence.restype = ctypes.c_int
    lib.oracle_gdn_frontend_head.argtypes = [i64, i64, i64, i64, i64, i64, i64,
                                             p, p, p, p, p, p, p, dbl,
                                             p, p, p, p, p]
    lib.oracle_gdn_frontend_head.restype = ctypes.c_int
    lib.oracle_conv_silu.argtypes = [i64, i64, i64, p, p, p, p]
    lib.oracle_conv_silu.restype = ctypes.c_int
    lib.oracle_gdn_layer.argtypes = [i64, i64, i64, i64, i64, p, p, p, p, p, p,
                                     p, i64, p, p, p, dbl, p, p, p, ctypes.c_int]
    lib.oracle_gdn_layer.restype = ctypes.c_int
    lib.oracle_gated_rmsnorm.argtypes = [i64, i64, p, p, p, dbl, p]
    lib.oracle_gate_projection.argtypes = [i64, i64, i64, p, p, p, p]
    lib.oracle_gate_projection.restype = ctypes.c_int
    lib.oracle_gated_rmsnorm.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def recurrence(qhat, khat, v, g, beta, S0=None):
    """Token-by-token gated delta rule for one head.

    qhat, khat: [T, d_k]; v: [T, d_v]; g, beta: [T]; S0: [d_v, d_k] (math
    layout, o = S q) or None.  Returns (o [T, d_v], S_T [d_v, d_k]).
    """
    lib = _load()
    qhat, khat, v, g, beta, S0 = map(_f64, (qhat, khat, v, g, beta, S0))
    T, d_k = qhat.shape
    d_v = v.shape[1]
    o = np.zeros((T, d_v), np.float64)
    S = np.zeros((d_v, d_k), np.float64)
    rc = lib.oracle_gdn_recurrence(T, d_k, d_v, _ptr(qhat), _ptr(khat), _ptr(v),
                                   _ptr(g), _ptr(beta), _ptr(S0), _ptr(o), _ptr(S))
    if rc:
        raise RuntimeError(f"oracle_gdn_recurrence failed ({rc})")
    return o, S


def frontend_head(x, a, b, conv_weight, A_log, dt_bias, h_k, h_v, d_k, d_v, h,
                  window0=None, l2_eps=L2_EPS):
    """Conv+SiLU, split, L2 norm (q also scaled by 1/sqrt(d_k)) and gates of one
    sequence for value head h.  Returns (qhat, khat, v, g, beta)."""
    lib = _load()
    x, a, b, conv_weight, A_log, dt_bias, window0 = map(
        _f32, (x, a, b, conv_weight, A_log, dt_bias, window0))
    T = x.shape[0]
    conv_w = conv_weight.shape[1]
    qh = np.zeros((T, d_k)); kh = np.zeros((T, d_k)); vv = np.zeros((T, d_v))
    g = np.zeros(T); be = np.zeros(T)
    rc = lib.oracle_gdn_frontend_head(T, h_k, h_v, d_k, d_v, conv_w, h, _ptr(x),
                                      _ptr(a), _ptr(b), _ptr(conv_weight),
                                      _ptr(A_log), _ptr(dt_bias), _ptr(window0),
                                      l2_eps, _ptr(qh), _ptr(kh), _ptr(vv),
                                      _ptr(g), _ptr(be))
    if rc:
        raise RuntimeError(f"oracle_gdn_frontend_head failed ({rc})")
    return qh, kh, vv, g, be


def conv_silu(x, conv_weight, window0=None):
    """Causal conv (tap W-1 on the current token) + SiLU of one sequence:
    x [T, conv_dim] -> y [T, conv_dim] float64."""
    lib = _load()
    x, conv_weight, window0 = map(_f32, (x, conv_weight, window0))
    T, conv_dim = x.shape
    y = np.zeros((T, conv_dim))
    rc = lib.oracle_conv_silu(T, conv_dim, conv_weight.shape[1], _ptr(x),
                              _ptr(window0), _ptr(conv_weight), _ptr(y))
    if rc:
        raise RuntimeError(f"oracle_conv_silu failed ({rc})")
    return y


def layer(x, a, b, conv_weight, A_log, dt_bias, cu_seqlens, h_k, h_v, d_k, d_v,
          window0=None, state0=None, head_mask=None, l2_eps=L2_EPS,
          n_threads=None, out=None):
    """Whole varlen Gated DeltaNet layer.

    x [T_tot, conv_dim]; a, b [T_tot, h_v]; cu_seqlens [B+1];
    window0 [B, W-1, conv_dim] or None; state0 [B, h_v, d_k, d_v] (S^T) or None;
    head_mask [B, h_v] bool or None.  Returns dict with o [T_tot, h_v, d_v],
    state [B, h_v, d_k, d_v] (S^T) and window [B, W-1, conv_dim], float64.
    """
    lib = _load()
    x, a, b, conv_weight, A_log, dt_bias, window0, state0 = map(
        _f32, (x, a, b, conv_weight, A_log, dt_bias, window0, state0))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    B = cu.shape[0] - 1
    T_tot, conv_dim = x.shape
    conv_w = conv_weight.shape[1]
    if out is None:
        out = {}
    o = out.get("o")
    if o is None:
        o = np.zeros((T_tot, h_v, d_v))
    st = out.get("state")
    if st is None:
        st = np.zeros((B, h_v, d_k, d_v))
    win = out.get("window")
    if win is None:
        win = np.zeros((B, conv_w - 1, conv_dim))
    mask = None if head_mask is None else np.ascontiguousarray(head_mask, dtype=np.uint8)
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    rc = lib.oracle_gdn_layer(h_k, h_v, d_k, d_v, conv_w, _ptr(x), _ptr(a), _ptr(b),
                              _ptr(conv_weight), _ptr(A_log), _ptr(dt_bias), _ptr(cu),
                              B, _ptr(window0), _ptr(state0), _ptr(mask), l2_eps,
                              _ptr(o), _ptr(st), _ptr(win), int(n_threads))
    if rc:
        raise RuntimeError(f"oracle_gdn_layer failed ({rc})")
    return {"o": o, "state": st, "window": win}


def slot_copy(state_pool, conv_pool, src, dst):
    """Snapshot / restore of recurrent state between slots (Vallmo.jl README,
    src/: the recurrent state is snapshotted and restored for prefix caching;
    PicoLM changelog, SSM State Checkpointing: capture and restore the full SSM
    state): for each pair i with src[i] >= 0 and dst[i] >= 0, slot dst[i]
    receives slot src[i]'s state and conv window.  Pairs apply in order;
    returns new float64 arrays."""
    st = np.array(state_pool, dtype=np.float64, copy=True)
    cw = np.array(conv_pool, dtype=np.float64, copy=True)
    for s_, d_ in zip(np.asarray(src).ravel(), np.asarray(dst).ravel()):
        if s_ >= 0 and d_ >= 0:
            st[d_] = st[s_]
            cw[d_] = cw[s_]
    return st, cw


def prefill_checkpoints(x, a, b, conv_weight, A_log, dt_bias, cu_seqlens, h_k, h_v, d_k, d_v,
                        every, window0=None, state0=None, l2_eps=L2_EPS):
    """Interval checkpoints of a prefill (PicoLM changelog, SSM State
    Checkpointing: checkpoints every N tokens during prefill; on reuse the
    closest one is restored and the remaining tokens are processed again).
    For sequence b and every k >= 1 with k * every < len_b: the state (S^T) and
    conv window after the first k * every tokens of the sequence, the
    sequence's initial state and window included -- by definition, the layer
    run on that prefix.  Returns a list over sequences of (states [n_b, h_v,
    d_k, d_v], windows [n_b, W-1, conv_dim]), n_b = ceil(len_b / every) - 1."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = cu.shape[0] - 1
    conv_dim = np.asarray(x).shape[1]
    conv_w = np.asarray(conv_weight).shape[1]
    out = []
    for bi in range(B):
        s0, ln = int(cu[bi]), int(cu[bi + 1] - cu[bi])
        n_b = max(0, -(-ln // every) - 1)
        states = np.zeros((n_b, h_v, d_k, d_v))
        windows = np.zeros((n_b, conv_w - 1, conv_dim))
        for k in range(1, n_b + 1):
            t = k * every
            r = layer(x[s0:s0 + t], a[s0:s0 + t], b[s0:s0 + t], conv_weight, A_log, dt_bias,
                      [0, t], h_k, h_v, d_k, d_v,
                      window0=None if window0 is None else window0[bi:bi + 1],
                      state0=None if state0 is None else state0[bi:bi + 1], l2_eps=l2_eps)
            states[k - 1] = r["state"][0]
            windows[k - 1] = r["window"][0]
        out.append((states, windows))
    return out


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))


def gated_rmsnorm(o, z, weight, eps=1e-6):
    """Gated RMSNorm of the layer output: o, z [..., d_v] -> y float64 with
    y = o / sqrt(mean(o^2) + eps) * weight * SiLU(z) over the last axis."""
    lib = _load()
    o, z, weight = map(_f32, (o, z, weight))
    shape = o.shape
    d_v = shape[-1]
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    y = np.zeros(shape)
    rc = lib.oracle_gated_rmsnorm(rows, d_v, _ptr(o), _ptr(z), _ptr(weight), float(eps), _ptr(y))
    if rc:
        raise RuntimeError(f"oracle_gated_rmsnorm failed ({rc})")
    return y


def gate_projection(hidden, w_ba, h_v):
    """The decay and beta input projections as one matmul: hidden [n][d_model]
    and w_ba [2 h_v][d_model] (decay rows first, then beta rows) -> (a, b),
    each [n][h_v] float64, a = hidden w_ba[:h_v]^T and b = hidden w_ba[h_v:]^T."""
    lib = _load()
    hidden, w_ba = _f32(hidden), _f32(w_ba)
    n, d_model = hidden.shape
    assert w_ba.shape == (2 * h_v, d_model)
    a = np.zeros((n, h_v))
    b = np.zeros((n, h_v))
    rc = lib.oracle_gate_projection(n, d_model, h_v, _ptr(hidden), _ptr(w_ba), _ptr(a), _ptr(b))
    if rc:
        raise RuntimeError(f"oracle_gate_projection failed ({rc})")
    return a, b
