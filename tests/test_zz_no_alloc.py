"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Code embedded in a host framework whose allocator already holds nearly all of
HBM, or running on a path where cudaMalloc's implicit synchronisation is not
acceptable, cannot allocate the workspace gdn_prefill wants; this entry point
uses a fixed scratch array inside the library's device image instead.

It runs the same kernels as gdn_prefill, so its results must equal
gdn_prefill's bit for bit, and both must match the float64 oracle.  The calls
here reuse the one shared scratch in an order meant to expose stale contents:
a long call, then a shorter one (fewer chunks, so the tail of the scratch
still holds the long call's records), then a call down the fp32-state SIMT
path (a different workspace layout over the same bytes).  A request larger
than the scratch must be refused before anything runs.

This file is collected last on purpose: it must pass run alone in a fresh
process and after the rest of the suite.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, TINY
from tests._gpu import PrefillRun, check_prefill, oracle_prefill

pytestmark = pytest.mark.gpu

FP32_STATE = dataclasses.replace(QWEN35_4B, flags=gdn.GDN_FP32_STATE)


def _noalloc(run):
    gdn.gdn_prefill_noalloc(run.dims, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b,
                            run.cu, run.slot, run.init, run.state, run.conv, run.o,
                            d_status=run.status)


def _largest_fitting(dims, lengths_of):
    """The largest n (a multiple of 64) for which lengths_of(n) still fits."""
    n = 64
    while gdn.gdn_prefill_workspace_size(dims, sum(lengths_of(n + 64)),
                                         len(lengths_of(n + 64))) <= gdn.GDN_NOALLOC_SCRATCH_BYTES:
        n += 64
    return n


def _calls():
    """(dims, lengths, seed) of the consecutive calls: long, then short, per path."""
    # the long tensor-core call nearly fills the scratch
    n = min(_largest_fitting(QWEN35_4B, lambda n: [n - 37, 37]), 2048)
    return [(QWEN35_4B, [n - 37, 37], 101),
            (QWEN35_4B, [300, 1, 64, 0, 130], 202),
            (FP32_STATE, [200, 77, 1], 303),
            (TINY, [64, 5, 17], 404),
            (TINY, [3], 505)]


def test_noalloc_prefill_equals_prefill_and_oracle_on_consecutive_calls(gpu_lib):
    for call, (dims, lengths, seed) in enumerate(_calls()):
        inp = workloads.layer_inputs(dims, lengths, seed=seed, init="mixed",
                                     num_slots=len(lengths) + 2)
        ref_run = PrefillRun(inp)     # the existing entry point, with its own workspace
        ref_run()
        ref = ref_run.results()
        run = PrefillRun(inp)         # fresh pools; the workspace it holds is not used
        _noalloc(run)
        got = run.results()
        what = f"call {call} ({lengths})"
        assert got["status"] == 0 and ref["status"] == 0, what
        # the same kernels on the same inputs: bit for bit
        np.testing.assert_array_equal(got["o"], ref["o"], err_msg=f"{what}: o")
        np.testing.assert_array_equal(got["state_pool"], ref["state_pool"],
                                      err_msg=f"{what}: state pool")
        np.testing.assert_array_equal(got["conv_pool"], ref["conv_pool"],
                                      err_msg=f"{what}: conv pool")
        # and against the oracle, so that a fault shared by both calls is caught
        check_prefill(inp, got, oracle_prefill(inp))


def test_noalloc_refuses_requests_beyond_its_scratch(gpu_lib):
    d = QWEN35_4B
    T = 64
    while gdn.gdn_prefill_workspace_size(d, T, 1) <= gdn.GDN_NOALLOC_SCRATCH_BYTES:
        T += 64   # the smallest multiple of 64 tokens that no longer fits
    inp = workloads.layer_inputs(d, [T], seed=5, init="random", num_slots=2)
    run = PrefillRun(inp)
    o_before = run.o.clone()
    state_before = run.state.clone()
    conv_before = run.conv.clone()
    with pytest.raises(gdn.GdnError) as exc:
        _noalloc(run)
    assert exc.value.status == -4  # GDN_EWORKSPACE
    torch.cuda.synchronize()
    # nothing ran: outputs, pools and the status word are as they were
    assert torch.equal(run.o.isnan(), o_before.isnan())
    assert torch.equal(run.state, state_before)
    assert torch.equal(run.conv, conv_before)
    assert run.status.item() == 0
