"""Prefill and decode at the same time: a prefill of three sequences on one
stream and a decode step over sixteen other slots of the same state and conv
pools on another, launched without waiting for each other, give bit for bit
the results of the two calls run one after the other (the layer-level
counterpart of serving prefill and decode requests concurrently)."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, TINY
from tests._gpu import dev, io_dtype

pytestmark = pytest.mark.gpu

NUM_SLOTS = 24


def _case(d):
    pre = workloads.layer_inputs(d, [300, 77, 129], seed=91, init="mixed", num_slots=NUM_SLOTS,
                                 shuffle_slots=False)            # slots 0, 1, 2
    dec = workloads.decode_inputs(d, n_rows=16, num_slots=NUM_SLOTS, seed=92)
    dec["slot_idx"] = (3 + np.random.default_rng(93).permutation(16)).astype(np.int32)
    return pre, dec


def _run(d, pre, dec, concurrent):
    io = io_dtype(d)
    state = dev(pre["state_pool"])
    conv = dev(pre["conv_pool"], io)
    T = pre["x"].shape[0]
    o_pre = torch.full((T, d.h_v, d.d_v), float("nan"), dtype=io, device="cuda")
    o_dec = torch.full((16, d.h_v, d.d_v), float("nan"), dtype=io, device="cuda")
    ws = torch.empty(gdn.gdn_prefill_workspace_size(d, T, 3), dtype=torch.uint8, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    args_pre = [dev(pre["conv_weight"]), dev(pre["A_log"]), dev(pre["dt_bias"]), dev(pre["x"], io),
                dev(pre["a"], io), dev(pre["b"], io), dev(pre["cu_seqlens"].astype(np.int32)),
                dev(pre["slot_idx"].astype(np.int32)), dev(pre["has_init"].astype(np.uint8))]
    args_dec = [dev(dec["conv_weight"]), dev(dec["A_log"]), dev(dec["dt_bias"]), dev(dec["x"], io),
                dev(dec["a"], io), dev(dec["b"], io), dev(dec["slot_idx"])]
    torch.cuda.synchronize()
    s1 = torch.cuda.Stream() if concurrent else torch.cuda.current_stream()
    s2 = torch.cuda.Stream() if concurrent else torch.cuda.current_stream()
    gdn.gdn_prefill(d, *args_pre, state, conv, o_pre, ws, d_status=status[0:1], stream=s1.cuda_stream)
    gdn.gdn_decode_step(d, *args_dec, state, conv, o_dec, d_status=status[1:2], stream=s2.cuda_stream)
    torch.cuda.synchronize()
    return {"o_pre": o_pre.float().cpu().numpy(), "o_dec": o_dec.float().cpu().numpy(),
            "state": state.cpu().numpy(), "conv": conv.float().cpu().numpy(),
            "status": status.cpu().numpy()}


@pytest.mark.parametrize("name", ["qwen35_4b", "tiny_fp32"])
def test_prefill_and_decode_on_two_streams_match_running_them_in_turn(gpu_lib, name):
    d = {"qwen35_4b": QWEN35_4B, "tiny_fp32": TINY}[name]
    pre, dec = _case(d)
    seq = _run(d, pre, dec, concurrent=False)
    con = _run(d, pre, dec, concurrent=True)
    assert not seq["status"].any() and not con["status"].any()
    for k in ("o_pre", "o_dec", "state", "conv"):
        assert np.isfinite(seq[k]).all(), k
        np.testing.assert_array_equal(con[k], seq[k], err_msg=k)
