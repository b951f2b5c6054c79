"""The bounded waits of the tensor-core prefill, made to run out.

Every wait between the prefill's CTAs and warps is bounded in global time
(%globaltimer).  GDN_TEST_WAIT_TIMEOUT (a test-only gdn_dims flag) shortens
the bound to 2 ms and has the prep kernel withhold the ready flag of the last
chunk of sequence 0, key head 0.  The scan CTAs of value heads 0 and 1 of
that sequence must then give up: GDN_DEV_WAIT_TIMEOUT set, their tensor
memory freed, no fault and no hang.  Everything that did not depend on the
withheld chunk is still right, and the next ordinary call on the same stream
runs clean.  Nothing here faults, traps or spins without a bound: the wait
that runs out is a sanctioned, short one.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B
from tests._gpu import PrefillRun, assert_close, check_prefill, oracle_prefill

pytestmark = pytest.mark.gpu


def test_withheld_chunk_times_out_and_the_next_call_is_clean(gpu_lib):
    inp = workloads.layer_inputs(QWEN35_4B, [300, 200], seed=31, init="random", num_slots=3)
    d_test = dataclasses.replace(QWEN35_4B, flags=gdn.GDN_TEST_WAIT_TIMEOUT)
    run = PrefillRun(dict(inp, dims=d_test))
    run()
    got = run.results()
    assert got["status"] & gdn.GDN_DEV_WAIT_TIMEOUT, got["status"]
    assert not got["status"] & ~gdn.GDN_DEV_WAIT_TIMEOUT, got["status"]
    ref = oracle_prefill(inp)
    cu = inp["cu_seqlens"]
    # what did not wait on the withheld chunk: sequence 1, and sequence 0's
    # value heads 2..31 (outputs and final states)
    for h in range(2, QWEN35_4B.h_v):
        assert_close(got["o"][cu[0]:cu[1], h], ref["o"][cu[0]:cu[1], h], QWEN35_4B, f"o seq 0 head {h}")
        assert_close(got["state_pool"][inp["slot_idx"][0], h], ref["state"][0, h], QWEN35_4B,
                     f"state seq 0 head {h}")
    for h in range(QWEN35_4B.h_v):
        assert_close(got["o"][cu[1]:cu[2], h], ref["o"][cu[1]:cu[2], h], QWEN35_4B, f"o seq 1 head {h}")
    # the next ordinary call on the same stream: clean status, right results
    run2 = PrefillRun(inp)
    run2()
    check_prefill(inp, run2.results(), ref)
    torch.cuda.synchronize()
