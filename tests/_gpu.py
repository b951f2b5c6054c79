"""Helpers of the GPU parity tests: run the CUDA path through the binding on a
workload dict (gated_deltanet_linear_07_gb300.workloads), run the oracle on
the same arrays, and compare with the stated tolerances.

Tolerances (per tensor kind, the max taken per (sequence, value head) block:
the outputs of one head over one sequence's tokens, or one head's final
state; per (row, value head) for decode):
  fp32 I/O:  |err| <= 1e-3 * max|ref| + 1e-5
  bf16 I/O:  |err| <= 2e-2 * max|ref|
Scoping the scale to a block keeps a wrong short sequence or a strongly
decayed head, whose values are small, from hiding under the batch's largest
values.  One exception: the outputs of a sequence shorter than one chunk (64
tokens) take the max over all of that sequence's heads.  There a head's
output can be a handful of tokens of beta v (q.k) with q nearly orthogonal to
k; the bf16 rounding of the normalised q and k (relative 2^-9 per element)
then leaves an error of ~2^-9 |q||k| / sqrt(d_k) on a dot product that is
itself much smaller, so the head's own max is no scale for it.
Integer and byte results (which slots were written, untouched slots, the conv
windows, which are raw copies of inputs) must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_linear_07_gb300 as gdn
import oracle
from gated_deltanet_linear_07_gb300 import workloads


def io_dtype(dims):
    return torch.bfloat16 if dims.io == "bf16" else torch.float32


def tol(dims):
    return (1e-3, 1e-5) if dims.io == "fp32" else (2e-2, 0.0)


def assert_close(got, ref, dims, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rel, ab = tol(dims)
    scale = np.abs(ref).max() if ref.size else 0.0
    err = np.abs(got - ref)
    bound = rel * scale + ab
    worst = float(err.max()) if err.size else 0.0
    assert worst <= bound, f"{what}: max err {worst:.3e} > {bound:.3e} (max|ref| {scale:.3e})"
    return worst / (scale if scale else 1.0)


def assert_close_heads(got, ref, dims, what, head_axis):
    """assert_close per value head: the scale of each head's block is its own
    max|ref|.  Returns the worst error normalised by its block's scale."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rel, ab = tol(dims)
    g = np.moveaxis(got, head_axis, 0).reshape(got.shape[head_axis], -1)
    r = np.moveaxis(ref, head_axis, 0).reshape(ref.shape[head_axis], -1)
    scale = np.abs(r).max(axis=1)
    err = np.abs(g - r).max(axis=1)
    bound = rel * scale + ab
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{what}: head {bad[0]} max err {err[bad[0]]:.3e} > "
                           f"{bound[bad[0]]:.3e} (max|ref| {scale[bad[0]]:.3e}; "
                           f"{bad.size} heads over)")
    return float((err / np.where(scale > 0, scale, 1.0)).max())


SHORT_SEQ = 64   # outputs of shorter sequences are scaled per sequence (see above)


def assert_close_seq_out(got, ref, dims, what):
    """One sequence's token-major outputs [T][h_v][d_v]: per value head, or
    over all heads when the sequence is shorter than SHORT_SEQ tokens."""
    if len(ref) < SHORT_SEQ:
        return assert_close(got, ref, dims, what)
    return assert_close_heads(got, ref, dims, what, head_axis=1)


def assert_close_seqs(got, ref, cu, dims, what):
    """Token-major outputs [T][h_v][d_v] of a varlen batch, checked per
    (sequence, value head) (per sequence when it is short)."""
    worst = 0.0
    for s in range(len(cu) - 1):
        lo, hi = int(cu[s]), int(cu[s + 1])
        worst = max(worst, assert_close_seq_out(got[lo:hi], ref[lo:hi], dims, f"{what} seq {s}"))
    return worst


def assert_close_rows(got, ref, dims, what):
    """Per-row tensors ([n][h_v][d_v] outputs or [n][h_v][d_k][d_v] states),
    checked per (row, value head)."""
    worst = 0.0
    for n in range(len(ref)):
        worst = max(worst, assert_close_heads(got[n], ref[n], dims, f"{what} {n}", head_axis=0))
    return worst


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device="cuda", dtype=dtype) if dtype is not None else t.cuda()


class PrefillRun:
    """Device copies of a prefill workload plus the call through the C ABI."""

    def __init__(self, inp):
        d = inp["dims"]
        self.inp, self.dims = inp, d
        io = io_dtype(d)
        self.x = dev(inp["x"], io)
        self.a = dev(inp["a"], io)
        self.b = dev(inp["b"], io)
        self.cw = dev(inp["conv_weight"])
        self.A_log = dev(inp["A_log"])
        self.dt_bias = dev(inp["dt_bias"])
        self.cu = dev(inp["cu_seqlens"].astype(np.int32))
        self.slot = dev(inp["slot_idx"].astype(np.int32))
        self.init = dev(inp["has_init"].astype(np.uint8))
        self.state = dev(inp["state_pool"])
        self.conv = dev(inp["conv_pool"], io)
        T = inp["x"].shape[0]
        self.o = torch.full((T, d.h_v, d.d_v), float("nan"), dtype=io, device="cuda")
        ws = gdn.gdn_prefill_workspace_size(d, T, len(inp["lengths"]))
        self.ws = torch.empty(max(ws, 1), dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def __call__(self, stream=None):
        gdn.gdn_prefill(self.dims, self.cw, self.A_log, self.dt_bias, self.x, self.a, self.b,
                        self.cu, self.slot, self.init, self.state, self.conv, self.o, self.ws,
                        d_status=self.status, stream=stream)

    def results(self):
        torch.cuda.synchronize()
        return {"o": self.o.float().cpu().numpy(), "state_pool": self.state.cpu().numpy(),
                "conv_pool": self.conv.float().cpu().numpy(), "status": int(self.status.item())}


def oracle_prefill(inp, head_mask=None, n_threads=None):
    d = inp["dims"]
    ov = workloads.oracle_view(inp)
    return oracle.layer(inp["x"], inp["a"], inp["b"], inp["conv_weight"], inp["A_log"],
                        inp["dt_bias"], inp["cu_seqlens"], d.h_k, d.h_v, d.d_k, d.d_v,
                        window0=ov["window0"], state0=ov["state0"], head_mask=head_mask,
                        l2_eps=d.l2_eps, n_threads=n_threads)


def check_prefill(inp, got, ref, head_mask=None):
    """Compare GPU prefill results with the oracle; returns the worst normalised error."""
    d = inp["dims"]
    B = len(inp["lengths"])
    cu = inp["cu_seqlens"]
    worst = 0.0
    if head_mask is None:
        for s in range(B):
            lo, hi = cu[s], cu[s + 1]
            worst = max(worst, assert_close_seq_out(got["o"][lo:hi], ref["o"][lo:hi], d,
                                                    f"o seq {s}"))
            worst = max(worst, assert_close_heads(got["state_pool"][inp["slot_idx"][s]],
                                                  ref["state"][s], d, f"state seq {s}",
                                                  head_axis=0))
    else:
        for s in range(B):
            for h in np.nonzero(head_mask[s])[0]:
                lo, hi = cu[s], cu[s + 1]
                worst = max(worst, assert_close(got["o"][lo:hi, h], ref["o"][lo:hi, h], d,
                                                f"o seq {s} head {h}"))
                worst = max(worst, assert_close(got["state_pool"][inp["slot_idx"][s], h],
                                                ref["state"][s, h], d, f"state seq {s} head {h}"))
    # windows are raw copies of inputs: exact
    for s in range(B):
        np.testing.assert_array_equal(got["conv_pool"][inp["slot_idx"][s]],
                                      ref["window"][s].astype(np.float32))
    # slots no sequence uses are untouched, bit for bit
    used = set(int(v) for v in inp["slot_idx"])
    for sl in range(inp["num_slots"]):
        if sl not in used:
            np.testing.assert_array_equal(got["state_pool"][sl], inp["state_pool"][sl])
            np.testing.assert_array_equal(got["conv_pool"][sl], inp["conv_pool"][sl])
    assert got["status"] == 0, got["status"]
    return worst


class DecodeRun:
    def __init__(self, inp):
        d = inp["dims"]
        self.inp, self.dims = inp, d
        io = io_dtype(d)
        self.x = dev(inp["x"], io)
        self.a = dev(inp["a"], io)
        self.b = dev(inp["b"], io)
        self.cw = dev(inp["conv_weight"])
        self.A_log = dev(inp["A_log"])
        self.dt_bias = dev(inp["dt_bias"])
        self.slot = dev(inp["slot_idx"].astype(np.int32))
        self.state = dev(inp["state_pool"])
        self.conv = dev(inp["conv_pool"], io)
        n = inp["x"].shape[0]
        self.o = torch.full((n, d.h_v, d.d_v), float("nan"), dtype=io, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def __call__(self, stream=None):
        gdn.gdn_decode_step(self.dims, self.cw, self.A_log, self.dt_bias, self.x, self.a, self.b,
                            self.slot, self.state, self.conv, self.o, d_status=self.status,
                            stream=stream)

    def results(self):
        torch.cuda.synchronize()
        return {"o": self.o.float().cpu().numpy(), "state_pool": self.state.cpu().numpy(),
                "conv_pool": self.conv.float().cpu().numpy(), "status": int(self.status.item())}


def oracle_decode(inp, rows=None):
    """Each decode row is a length-1 sequence starting from its slot's state and window."""
    d = inp["dims"]
    sl = inp["slot_idx"]
    rows = [n for n in range(len(sl)) if sl[n] >= 0] if rows is None else list(rows)
    r = oracle.layer(inp["x"][rows], inp["a"][rows], inp["b"][rows], inp["conv_weight"],
                     inp["A_log"], inp["dt_bias"], np.arange(len(rows) + 1), d.h_k, d.h_v,
                     d.d_k, d.d_v, window0=inp["conv_pool"][sl[rows]],
                     state0=inp["state_pool"][sl[rows]], l2_eps=d.l2_eps)
    r["rows"] = rows
    return r


def check_decode(inp, got, ref):
    d = inp["dims"]
    rows = ref["rows"]
    sl = inp["slot_idx"]
    worst = 0.0
    for i, n in enumerate(rows):   # per (row, value head)
        worst = max(worst, assert_close_heads(got["o"][n], ref["o"][i], d, f"decode o row {n}",
                                              head_axis=0))
        worst = max(worst, assert_close_heads(got["state_pool"][sl[n]], ref["state"][i], d,
                                              f"decode state row {n}", head_axis=0))
    np.testing.assert_array_equal(got["conv_pool"][sl[rows]], ref["window"].astype(np.float32))
    pad = [n for n in range(len(sl)) if sl[n] < 0]
    if pad:
        assert not got["o"][pad].any(), "padding rows must be zero"
    used = set(int(v) for v in sl if v >= 0)
    for s in range(inp["num_slots"]):
        if s not in used:
            np.testing.assert_array_equal(got["state_pool"][s], inp["state_pool"][s])
            np.testing.assert_array_equal(got["conv_pool"][s], inp["conv_pool"][s])
    return worst
