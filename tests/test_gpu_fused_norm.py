"""GPU parity of the layer with the gated RMSNorm of its output
(gdn_prefill_gated_norm, gdn_decode_step_gated_norm, called through the C ABI)
against the float64 oracle, within the stated tolerances of tests/_gpu.py.
The states and windows these calls leave are bit for bit those of the plain
calls, since the norm touches only the output; the tensor-core and SIMT
prefill paths (varlen, mixed initial states) and the decode step, whose
epilogue computes the norm itself, with padding rows, are covered.

Prefill is checked stage by stage: the plain call's o against the oracle's
layer, and the fused call's y against the oracle's norm of that same o.  The
norm rescales every (token, head) row to unit RMS, so a row whose bf16 output
is a small difference (the first tokens of a sequence, q nearly orthogonal to
k) carries the layer's rounding into y at full scale; comparing y with the
oracle's norm of the oracle's o would test that rounding a second time.  The
decode step works in fp32 throughout and is compared end to end."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
import oracle
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, TINY, Dims
from tests._gpu import (DecodeRun, PrefillRun, assert_close, assert_close_rows, assert_close_seqs,
                        check_prefill, dev, io_dtype, oracle_decode, oracle_prefill)

pytestmark = pytest.mark.gpu

PREFILL = {
    "qwen35_4b": (QWEN35_4B, [130, 64, 300, 1, 77]),        # tensor-core path
    "tiny_fp32": (TINY, [64, 9, 33]),                       # SIMT path
    "asym_bf16": (Dims(h_k=1, h_v=2, d_k=16, d_v=32, chunk=32, io="bf16"), [100, 31]),
}


def _gate_inputs(d, T, seed):
    rng = np.random.default_rng(seed)
    z = (2.0 * rng.standard_normal((T, d.h_v, d.d_v))).astype(np.float32)
    z[-1, :, : d.d_v // 2] = 30.0                         # open and closed gates
    z[-1, :, d.d_v // 2:] = -30.0
    w = rng.uniform(0.25, 2.0, d.d_v).astype(np.float32)
    if d.io == "bf16":
        z = workloads.round_bf16(z)
    return z, w


@pytest.mark.parametrize("name", sorted(PREFILL))
def test_fused_prefill_matches_oracle(gpu_lib, name):
    d, lengths = PREFILL[name]
    inp = workloads.layer_inputs(d, lengths, seed=60 + len(name), init="mixed")
    T = inp["x"].shape[0]
    z, w = _gate_inputs(d, T, seed=61)
    plain = PrefillRun(inp)
    plain()
    base = plain.results()
    run = PrefillRun(inp)
    dz = dev(z, io_dtype(d))
    gdn.gdn_prefill_gated_norm(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu,
                               run.slot, run.init, run.state, run.conv, dz, dev(w), run.o, run.ws,
                               eps=1e-6, d_status=run.status)
    got = run.results()
    assert got["status"] == 0
    np.testing.assert_array_equal(got["state_pool"], base["state_pool"])
    np.testing.assert_array_equal(got["conv_pool"], base["conv_pool"])
    np.testing.assert_array_equal(dz.float().cpu().numpy(), z)          # z is not touched
    check_prefill(inp, base, oracle_prefill(inp))        # the layer
    ref = oracle.gated_rmsnorm(base["o"], z, w, eps=1e-6)  # the norm of its o
    worst = assert_close_seqs(got["o"], ref, inp["cu_seqlens"], d, f"{name} y")
    print(f"fused prefill {name}: worst normalised error {worst:.3e}")


def test_fused_prefill_qwen35_4b_full_size_sampled(gpu_lib):
    """The T=4096 Qwen3.5-4B prefill with the norm fused: 6 sampled value heads
    against the oracle, every token."""
    inp = workloads.prefill_4b()
    d = inp["dims"]
    T = inp["x"].shape[0]
    z, w = _gate_inputs(d, T, seed=62)
    plain = PrefillRun(inp)
    plain()
    base = plain.results()
    run = PrefillRun(inp)
    gdn.gdn_prefill_gated_norm(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu,
                               run.slot, run.init, run.state, run.conv, dev(z, torch.bfloat16),
                               dev(w), run.o, run.ws, d_status=run.status)
    got = run.results()
    assert got["status"] == 0
    heads = np.random.default_rng(8).choice(d.h_v, 6, replace=False)
    mask = np.zeros((len(inp["lengths"]), d.h_v), bool)
    mask[:, heads] = True
    ref = oracle_prefill(inp, head_mask=mask)
    cu = inp["cu_seqlens"]
    for s in range(len(inp["lengths"])):
        for h in heads:
            lo, hi = cu[s], cu[s + 1]
            assert_close(base["o"][lo:hi, h], ref["o"][lo:hi, h], d, f"o seq {s} head {h}")
            y = oracle.gated_rmsnorm(base["o"][lo:hi, h], z[lo:hi, h], w)
            assert_close(got["o"][lo:hi, h], y, d, f"y seq {s} head {h}")


@pytest.mark.parametrize("name", ["qwen35_4b", "tiny_fp32", "asym_bf16"])
def test_fused_decode_matches_oracle(gpu_lib, name):
    d = PREFILL[name][0]
    inp = workloads.decode_inputs(d, n_rows=24, num_slots=40, seed=63, padding_rows=2)
    z, w = _gate_inputs(d, 24, seed=64)
    plain = DecodeRun(inp)
    plain()
    base = plain.results()
    run = DecodeRun(inp)
    gdn.gdn_decode_step_gated_norm(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b,
                                   run.slot, run.state, run.conv, dev(z, io_dtype(d)), dev(w),
                                   run.o, eps=1e-6, d_status=run.status)
    got = run.results()
    assert got["status"] == 0
    np.testing.assert_array_equal(got["state_pool"], base["state_pool"])
    np.testing.assert_array_equal(got["conv_pool"], base["conv_pool"])
    ref = oracle_decode(inp)
    rows = ref["rows"]
    y = oracle.gated_rmsnorm(ref["o"], z[rows], w, eps=1e-6)
    worst = assert_close_rows(got["o"][rows], y, d, f"{name} decode y row")
    pad = [n for n in range(24) if inp["slot_idx"][n] < 0]
    assert pad and not got["o"][pad].any(), "padding rows must be zero"
    print(f"fused decode {name}: worst normalised error {worst:.3e}")
