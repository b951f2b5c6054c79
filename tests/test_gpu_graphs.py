"""The library's calls inside CUDA graphs: gdn_prefill (tensor-core path, its
set-up, prep and scan launches with their programmatic dependencies; and the
SIMT path) and a run of decode steps, captured once with torch.cuda.CUDAGraph
and replayed, give bit for bit the results of the plain calls on the same
inputs.  The kernels have fixed reduction orders, so any difference would mean
a launch that depends on host state the graph froze (a pointer, a size, a
tensor map) or an ordering the capture lost."""
import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, Dims
from tests._gpu import DecodeRun, PrefillRun

pytestmark = pytest.mark.gpu


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    torch.cuda.synchronize()
    return g


def _snapshot(run):
    torch.cuda.synchronize()
    return {"o": run.o.clone(), "state": run.state.clone(), "conv": run.conv.clone(),
            "status": run.status.clone()}


def _restore(run, snap0):
    run.o.fill_(float("nan"))
    run.state.copy_(snap0["state"])
    run.conv.copy_(snap0["conv"])
    run.status.zero_()


def _assert_same(a, b):
    for k in ("o", "state", "conv", "status"):
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k


PREFILL_CASES = {
    "qwen35_4b_tensor_cores": (QWEN35_4B, [300, 77, 0, 129]),
    "qwen35_4b_fp32_state_simt": (dataclasses.replace(QWEN35_4B, flags=gdn.GDN_FP32_STATE), [130, 5]),
    "small_simt_fp32": (Dims(h_k=2, h_v=4, d_k=32, d_v=16, chunk=32, io="fp32"), [70, 1, 33]),
}


@pytest.mark.parametrize("name", list(PREFILL_CASES))
def test_prefill_replayed_from_a_graph_matches_the_plain_call(gpu_lib, name):
    d, lengths = PREFILL_CASES[name]
    inp = workloads.layer_inputs(d, lengths, seed=4242, init="mixed", num_slots=len(lengths) + 3)
    run = PrefillRun(inp)
    snap0 = _snapshot(run)
    run()
    plain = _snapshot(run)
    assert plain["status"].item() == 0
    _restore(run, snap0)
    g = _capture(run)               # the capture's own warm-up call ran on a side stream
    for _ in range(2):              # replays from the same initial pools
        _restore(run, snap0)
        g.replay()
        _assert_same(plain, _snapshot(run))


def test_decode_steps_replayed_from_a_graph_match_the_plain_calls(gpu_lib):
    d = QWEN35_4B
    inp = workloads.decode_inputs(d, n_rows=12, num_slots=16, seed=4343, padding_rows=2)
    run = DecodeRun(inp)
    snap0 = _snapshot(run)

    def three_steps():              # the same rows three times: each step reads the last one's state
        for _ in range(3):
            run()

    three_steps()
    plain = _snapshot(run)
    assert plain["status"].item() == 0
    assert not np.isnan(plain["o"].float().cpu().numpy()).all()
    _restore(run, snap0)
    g = _capture(three_steps)
    _restore(run, snap0)
    g.replay()
    _assert_same(plain, _snapshot(run))
