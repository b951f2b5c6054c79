"""GPU parity of slot copies (gdn_slot_copy) and interval checkpoints
(gdn_prefill_checkpointed), called through the C ABI, against the float64
oracle: copies are exact; checkpoint states within the stated tolerances of
tests/_gpu.py, checkpoint windows exact; the layer's own outputs and final
states bit for bit those of gdn_prefill; every slot the call does not name is
untouched; a prefill resumed from a checkpoint slot continues the sequence."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
import oracle
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, TINY, Dims
from tests._gpu import PrefillRun, assert_close, assert_close_heads, dev, io_dtype

pytestmark = pytest.mark.gpu

SHAPES = {
    "qwen35_4b": (QWEN35_4B, [130, 64, 300, 1], 64),      # tensor-core path, chunk 64
    "qwen35_4b_every128": (QWEN35_4B, [257, 128], 128),
    "tiny_fp32": (TINY, [64, 9, 33], 16),                 # SIMT path, chunk 16
    "asym_bf16": (Dims(h_k=1, h_v=2, d_k=16, d_v=32, chunk=32, io="bf16"), [100, 31], 32),
    # SIMT path, chunk 128: checkpoints land after every 128-token chunk
    "c128_bf16": (Dims(h_k=1, h_v=2, d_k=32, d_v=32, chunk=128, io="bf16"), [300, 129, 1], 128),
}


def _n_ckpt(length, every):
    return max(0, -(-length // every) - 1)


# ---------------------------------------------------------------- slot copy

@pytest.mark.parametrize("name", ["qwen35_4b", "tiny_fp32"])
def test_slot_copy_matches_oracle(gpu_lib, name):
    d = SHAPES[name][0]
    inp = workloads.layer_inputs(d, [8], seed=31, num_slots=8)
    st, cw = dev(inp["state_pool"]), dev(inp["conv_pool"], io_dtype(d))
    src, dst = [1, 5, -1, 6, 2], [3, 0, 2, 6, -1]       # padding pairs, a self copy
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_slot_copy(d, st, cw, dev(np.array(src, np.int32)), dev(np.array(dst, np.int32)),
                      d_status=status)
    torch.cuda.synchronize()
    ref_st, ref_cw = oracle.slot_copy(inp["state_pool"], inp["conv_pool"], src, dst)
    np.testing.assert_array_equal(st.cpu().numpy(), ref_st.astype(np.float32))
    np.testing.assert_array_equal(cw.float().cpu().numpy(), ref_cw.astype(np.float32))
    assert status.item() == 0


def test_slot_copy_out_of_range_sets_status_and_copies_nothing(gpu_lib):
    d = QWEN35_4B
    inp = workloads.layer_inputs(d, [8], seed=32, num_slots=4)
    st, cw = dev(inp["state_pool"]), dev(inp["conv_pool"], io_dtype(d))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_slot_copy(d, st, cw, dev(np.array([0, 4], np.int32)), dev(np.array([4, 1], np.int32)),
                      d_status=status)
    torch.cuda.synchronize()
    assert status.item() & gdn.GDN_DEV_BAD_SLOT
    np.testing.assert_array_equal(st.cpu().numpy(), inp["state_pool"])
    np.testing.assert_array_equal(cw.float().cpu().numpy(), inp["conv_pool"].astype(np.float32))


# ---------------------------------------------------------------- checkpoints

def _ckpt_case(name, seed):
    """Sequences in slots B-1, ..., 0 (reversed); sequence s's checkpoints in the
    consecutive slots after them, s by s; two spare slots at the end."""
    d, lengths, every = SHAPES[name]
    n_ck = [_n_ckpt(t, every) for t in lengths]
    B = len(lengths)
    num_slots = B + sum(n_ck) + 2
    inp = workloads.layer_inputs(d, lengths, seed=seed, init="mixed", num_slots=num_slots,
                                 shuffle_slots=False)
    inp["slot_idx"] = np.arange(B - 1, -1, -1, dtype=np.int32)
    ck_slot = np.cumsum([B] + n_ck[:-1]).astype(np.int32)
    ck_slot[np.array(n_ck) == 0] = -1
    return inp, every, ck_slot, n_ck


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_checkpointed_prefill_matches_oracle(gpu_lib, name):
    inp, every, ck_slot, n_ck = _ckpt_case(name, seed=40 + len(name))
    d = inp["dims"]
    # the plain prefill, for the bit-for-bit comparison of the layer's own results
    plain = PrefillRun(inp)
    plain()
    base = plain.results()
    run = PrefillRun(inp)
    gdn.gdn_prefill_checkpointed(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu,
                                 run.slot, run.init, run.state, run.conv, run.o, run.ws, every,
                                 dev(ck_slot), d_status=run.status)
    got = run.results()
    assert got["status"] == 0, got["status"]
    np.testing.assert_array_equal(got["o"], base["o"])
    for s in inp["slot_idx"]:
        np.testing.assert_array_equal(got["state_pool"][s], base["state_pool"][s])
        np.testing.assert_array_equal(got["conv_pool"][s], base["conv_pool"][s])
    ov = workloads.oracle_view(inp)
    ref = oracle.prefill_checkpoints(inp["x"], inp["a"], inp["b"], inp["conv_weight"], inp["A_log"],
                                     inp["dt_bias"], inp["cu_seqlens"], d.h_k, d.h_v, d.d_k, d.d_v,
                                     every, window0=ov["window0"], state0=ov["state0"],
                                     l2_eps=d.l2_eps)
    named = set(int(s) for s in inp["slot_idx"])
    for s, (states, windows) in enumerate(ref):
        assert states.shape[0] == n_ck[s]
        for k in range(n_ck[s]):
            sl = int(ck_slot[s]) + k
            named.add(sl)
            assert_close_heads(got["state_pool"][sl], states[k], d, f"checkpoint {k} of seq {s}",
                               head_axis=0)
            np.testing.assert_array_equal(got["conv_pool"][sl], windows[k].astype(np.float32))
    for sl in range(inp["num_slots"]):
        if sl not in named:
            np.testing.assert_array_equal(got["state_pool"][sl], inp["state_pool"][sl])
            np.testing.assert_array_equal(got["conv_pool"][sl], inp["conv_pool"][sl])


def test_prefill_resumed_from_a_checkpoint_continues_the_sequence(gpu_lib):
    """Prefill 300 tokens with checkpoints every 64; then a prefill of tokens
    [128, 300) from checkpoint 2's slot gives the full run's outputs for them
    and its final state."""
    d = QWEN35_4B
    inp = workloads.layer_inputs(d, [300], seed=45, init="random", num_slots=8,
                                 shuffle_slots=False)    # the sequence in slot 0
    run = PrefillRun(inp)
    ck_slot = np.array([4], np.int32)                     # checkpoints 1..4 in slots 4..7
    gdn.gdn_prefill_checkpointed(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu,
                                 run.slot, run.init, run.state, run.conv, run.o, run.ws, 64,
                                 dev(ck_slot), d_status=run.status)
    full = run.results()
    assert full["status"] == 0
    # resume: tokens [128, 300) from slot 5 (checkpoint 2, after 128 tokens)
    t0 = 128
    T2 = 300 - t0
    io = io_dtype(d)
    o2 = torch.full((T2, d.h_v, d.d_v), float("nan"), dtype=io, device="cuda")
    ws = torch.empty(gdn.gdn_prefill_workspace_size(d, T2, 1), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill(d, run.cw, run.A_log, run.dt_bias, run.x[t0:], run.a[t0:], run.b[t0:],
                    dev(np.array([0, T2], np.int32)), dev(np.array([5], np.int32)),
                    dev(np.array([1], np.uint8)), run.state, run.conv, o2, ws, d_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert_close_heads(o2.float().cpu().numpy(), full["o"][t0:], d, "resumed o", head_axis=1)
    assert_close_heads(run.state[5].cpu().numpy(), full["state_pool"][0], d, "resumed final state",
                       head_axis=0)


def test_checkpoint_slot_out_of_range_sets_status(gpu_lib):
    d = QWEN35_4B
    inp = workloads.layer_inputs(d, [200], seed=46, num_slots=3, shuffle_slots=False)
    run = PrefillRun(inp)
    gdn.gdn_prefill_checkpointed(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu,
                                 run.slot, run.init, run.state, run.conv, run.o, run.ws, 64,
                                 dev(np.array([2], np.int32)), d_status=run.status)
    got = run.results()
    # checkpoints 1..3 would go to slots 2, 3, 4: slots 3 and 4 do not exist
    assert got["status"] & gdn.GDN_DEV_BAD_SLOT
    assert np.isfinite(got["o"]).all()


def test_checkpointed_prefill_full_size_sampled(gpu_lib):
    """The T=4096 Qwen3.5-4B prefill with a checkpoint every 256 tokens (15 of
    them, the bench's configuration): checkpoints 1, 8 and 15 against the
    oracle on the prefix, on 6 sampled value heads; their windows exact."""
    inp = workloads.prefill_4b()
    d = inp["dims"]
    every, n_ck = 256, 15
    base = inp["num_slots"]
    inp["state_pool"] = np.concatenate(
        [inp["state_pool"], np.zeros((n_ck,) + inp["state_pool"].shape[1:], np.float32)])
    inp["conv_pool"] = np.concatenate(
        [inp["conv_pool"], np.zeros((n_ck,) + inp["conv_pool"].shape[1:], np.float32)])
    inp["num_slots"] = base + n_ck
    run = PrefillRun(inp)
    gdn.gdn_prefill_checkpointed(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu,
                                 run.slot, run.init, run.state, run.conv, run.o, run.ws, every,
                                 dev(np.array([base], np.int32)), d_status=run.status)
    got = run.results()
    assert got["status"] == 0
    heads = np.random.default_rng(7).choice(d.h_v, 6, replace=False)
    mask = np.zeros((1, d.h_v), bool)
    mask[0, heads] = True
    for k in (1, 8, 15):
        t = k * every
        ref = oracle.layer(inp["x"][:t], inp["a"][:t], inp["b"][:t], inp["conv_weight"],
                           inp["A_log"], inp["dt_bias"], [0, t], d.h_k, d.h_v, d.d_k, d.d_v,
                           head_mask=mask, l2_eps=d.l2_eps)
        sl = base + k - 1
        for h in heads:
            assert_close(got["state_pool"][sl, h], ref["state"][0, h], d,
                         f"checkpoint {k} head {h}")
        np.testing.assert_array_equal(got["conv_pool"][sl], inp["x"][t - 3:t].astype(np.float32))
