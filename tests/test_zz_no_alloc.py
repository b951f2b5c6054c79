"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Code embedded in a host framework whose allocator already holds nearly all of
HBM, or running on a path where cudaMalloc's implicit synchronisation is not
acceptable, cannot allocate the workspace gdn_prefill wants; this entry point
uses a fixed scratch array inside the library's device image instead.  Its
results must equal gdn_prefill's (same kernels, same tolerance as every other
parity test here) on consecutive calls that reuse the shared scratch, and a
request larger than the scratch must be refused before anything runs.

This file is collected last on purpose: it must pass run alone in a fresh
process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, TINY
from tests._gpu import PrefillRun, assert_close

pytestmark = pytest.mark.gpu


def _noalloc(run):
    gdn.gdn_prefill_noalloc(run.dims, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b,
                            run.cu, run.slot, run.init, run.state, run.conv, run.o,
                            d_status=run.status)


@pytest.mark.parametrize("dims,lengths", [(QWEN35_4B, [300, 1, 64, 500, 0, 130]),
                                          (TINY, [64, 5, 17])])
def test_noalloc_prefill_matches_prefill_on_two_calls_in_a_row(gpu_lib, dims, lengths):
    for call, seed in enumerate((101, 202)):
        inp = workloads.layer_inputs(dims, lengths, seed=seed, init="mixed",
                                     num_slots=len(lengths) + 2)
        ref_run = PrefillRun(inp)     # the existing entry point, with its own workspace
        ref_run()
        ref = ref_run.results()
        run = PrefillRun(inp)         # fresh pools; the workspace it holds is not used
        _noalloc(run)
        got = run.results()
        assert got["status"] == 0 and ref["status"] == 0
        assert_close(got["o"], ref["o"], dims, f"call {call}: o")
        assert_close(got["state_pool"], ref["state_pool"], dims, f"call {call}: state pool")
        np.testing.assert_array_equal(got["conv_pool"], ref["conv_pool"])


def test_noalloc_refuses_requests_beyond_its_scratch(gpu_lib):
    d = QWEN35_4B
    T = 64
    while gdn.gdn_prefill_workspace_size(d, T, 1) <= gdn.GDN_NOALLOC_SCRATCH_BYTES:
        T += 64   # the smallest multiple of 64 tokens that no longer fits
    inp = workloads.layer_inputs(d, [T], seed=5, init="zero", num_slots=1)
    run = PrefillRun(inp)
    o_before = run.o.clone()
    with pytest.raises(gdn.GdnError) as exc:
        _noalloc(run)
    assert exc.value.status == -4  # GDN_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(run.o.isnan(), o_before.isnan())  # nothing ran
