"""GPU parity: the CUDA path, called through the C ABI, against the float64
oracle on identical seeded inputs, element by element, with the tolerances in
tests/_gpu.py.  Sizes span several chunks with ragged tails; the Qwen3.5-4B
prefill (T=4096) and the 24-layer x 64-slot decode step run at full size in
the launch configuration the benchmark times."""
import dataclasses
import os
import zlib

import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, TINY, Dims
from tests._gpu import (DecodeRun, PrefillRun, check_decode, check_prefill, dev, io_dtype,
                        oracle_decode, oracle_prefill)
import oracle

pytestmark = pytest.mark.gpu

NCPU = os.cpu_count() or 1


def test_tiny_prefill_matches_oracle(gpu_lib):
    inp = workloads.tiny()
    run = PrefillRun(inp)
    run()
    check_prefill(inp, run.results(), oracle_prefill(inp))


def test_tiny_token_by_token_decode_matches_prefill_oracle(gpu_lib):
    """The tiny workload fed one token at a time through the decode step equals
    the oracle's recurrence over the whole sequence."""
    inp = workloads.tiny()
    d = inp["dims"]
    ref = oracle_prefill(inp)
    io = io_dtype(d)
    state = torch.zeros((1, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device="cuda")
    conv = torch.zeros((1, 3, d.conv_dim), dtype=io, device="cuda")
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    cw, A, dt = dev(inp["conv_weight"]), dev(inp["A_log"]), dev(inp["dt_bias"])
    outs = []
    for t in range(inp["x"].shape[0]):
        o = torch.empty((1, d.h_v, d.d_v), dtype=io, device="cuda")
        gdn.gdn_decode_step(d, cw, A, dt, dev(inp["x"][t:t + 1], io), dev(inp["a"][t:t + 1], io),
                            dev(inp["b"][t:t + 1], io), slot, state, conv, o)
        outs.append(o)
    got = torch.cat(outs).float().cpu().numpy()
    from tests._gpu import assert_close_heads
    assert_close_heads(got, ref["o"], d, "o", head_axis=1)
    assert_close_heads(state[0].cpu().numpy(), ref["state"][0], d, "state", head_axis=0)
    np.testing.assert_array_equal(conv[0].float().cpu().numpy(), ref["window"][0])


LENGTHS = [0, 1, 2, 3, 15, 16, 17, 63, 64, 65, 130, 200]
SHAPES = {
    "asym_fp32": Dims(h_k=2, h_v=4, d_k=32, d_v=64, chunk=16, io="fp32"),
    "asym2_bf16": Dims(h_k=1, h_v=2, d_k=16, d_v=32, chunk=32, io="bf16"),
    "tall_fp32": Dims(h_k=1, h_v=1, d_k=128, d_v=16, chunk=64, io="fp32"),
    # chunk 128 (the SIMT path; at head dim 128 its scan streams the chunk inputs)
    "c128_bf16": Dims(h_k=2, h_v=4, d_k=64, d_v=64, chunk=128, io="bf16"),
    "c128_fp32": Dims(h_k=1, h_v=2, d_k=32, d_v=16, chunk=128, io="fp32"),
    "qwen35_4b_c128": dataclasses.replace(QWEN35_4B, chunk=128),
    "qwen35_4b": QWEN35_4B,
    # the tensor-core path with bf16 instead of fp16 MMA operands
    "qwen35_4b_bf16_ops": dataclasses.replace(QWEN35_4B, flags=gdn.GDN_BF16_OPERANDS),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("init", ["zero", "mixed", "random"])
def test_prefill_varlen_matches_oracle(gpu_lib, name, init):
    d = SHAPES[name]
    inp = workloads.layer_inputs(d, LENGTHS, seed=zlib.crc32(f"{name}-{init}".encode()) % 10000, init=init,
                                 num_slots=len(LENGTHS) + 3)
    run = PrefillRun(inp)
    run()
    check_prefill(inp, run.results(), oracle_prefill(inp, n_threads=NCPU))


def test_prefill_chunk128_spans_several_chunks(gpu_lib):
    """Chunk 128 over sequences of three, two and one chunks (ragged tails),
    with random initial states: the chunk-local factors and the cross-chunk
    scan at the largest chunk length."""
    d = SHAPES["c128_bf16"]
    inp = workloads.layer_inputs(d, [300, 256, 129, 1, 0], seed=128, init="random")
    run = PrefillRun(inp)
    run()
    check_prefill(inp, run.results(), oracle_prefill(inp, n_threads=NCPU))


def test_prefill_correlated_keys_stay_finite_and_match(gpu_lib):
    """Fully correlated keys (runs of one repeated key) with beta near 1 and no
    decay: the chunk inverse has entries -b(1-b)^m that a matrix-power scheme
    would blow up; exact substitution stays finite and matches the oracle."""
    inp = workloads.layer_inputs(QWEN35_4B, [700, 300], seed=44, init="random",
                                 b_mean=6.0, a_const=-12.0, correlated_keys=128)
    run = PrefillRun(inp)
    run()
    check_prefill(inp, run.results(), oracle_prefill(inp, n_threads=NCPU))


@pytest.mark.parametrize("name", sorted(SHAPES) + ["tiny"])
def test_decode_matches_oracle(gpu_lib, name):
    d = TINY if name == "tiny" else SHAPES[name]
    inp = workloads.decode_inputs(d, n_rows=12, num_slots=20, seed=77, padding_rows=2)
    run = DecodeRun(inp)
    run()
    check_decode(inp, run.results(), oracle_decode(inp))


def test_decode_is_bitwise_independent_of_row_order(gpu_lib):
    """A slot's result does not depend on which row carries it or on the rest of
    the batch: byte-identical batched-vs-single decode (oxydllm notes, New
    Features: the adversarial battery checks that)."""
    inp = workloads.decode_inputs(QWEN35_4B, n_rows=16, num_slots=16, seed=5)
    r1 = DecodeRun(inp)
    r1()
    g1 = r1.results()
    perm = np.random.default_rng(1).permutation(16)
    inp2 = dict(inp, x=inp["x"][perm], a=inp["a"][perm], b=inp["b"][perm],
                slot_idx=inp["slot_idx"][perm])
    r2 = DecodeRun(inp2)
    r2()
    g2 = r2.results()
    assert np.array_equal(g1["o"][perm], g2["o"])
    assert np.array_equal(g1["state_pool"], g2["state_pool"])
    single = dict(inp, x=inp["x"][3:4], a=inp["a"][3:4], b=inp["b"][3:4],
                  slot_idx=inp["slot_idx"][3:4])
    r3 = DecodeRun(single)
    r3()
    g3 = r3.results()
    assert np.array_equal(g3["o"][0], g1["o"][3])
    s = inp["slot_idx"][3]
    assert np.array_equal(g3["state_pool"][s], g1["state_pool"][s])


def test_conv1d_update_matches_oracle(gpu_lib):
    for d in (QWEN35_4B, TINY):
        inp = workloads.decode_inputs(d, n_rows=6, num_slots=9, seed=3, padding_rows=1)
        io = io_dtype(d)
        x, conv = dev(inp["x"], io), dev(inp["conv_pool"], io)
        y = torch.full((6, d.conv_dim), float("nan"), dtype=io, device="cuda")
        slot = dev(inp["slot_idx"])
        gdn.gdn_conv1d_update(d, dev(inp["conv_weight"]), x, conv, slot, y)
        torch.cuda.synchronize()
        y = y.float().cpu().numpy()
        conv = conv.float().cpu().numpy()
        for n, s in enumerate(inp["slot_idx"]):
            if s < 0:
                assert not y[n].any()
                continue
            ref = oracle.conv_silu(inp["x"][n:n + 1], inp["conv_weight"], inp["conv_pool"][s])
            from tests._gpu import assert_close
            assert_close(y[n:n + 1], ref, d, "conv y")
            hist = np.concatenate([inp["conv_pool"][s], inp["x"][n:n + 1]])
            np.testing.assert_array_equal(conv[s], hist[1:])


def test_prefill_then_prefill_then_decode_handoff(gpu_lib):
    """prefill(T1) -> prefill(T2, initial state from the slot) -> decode steps
    equals one oracle recurrence over all tokens (oxydllm notes, Tests:
    prefill-to-decode handoff)."""
    d = QWEN35_4B
    full = workloads.layer_inputs(d, [150], seed=8, init="random", num_slots=3)
    T1 = 70
    ref = oracle_prefill(full, n_threads=NCPU)
    io = io_dtype(d)
    state = dev(full["state_pool"])
    conv = dev(full["conv_pool"], io)
    cw, A, dt = dev(full["conv_weight"]), dev(full["A_log"]), dev(full["dt_bias"])
    slot = dev(full["slot_idx"])
    one = torch.ones(1, dtype=torch.uint8, device="cuda")
    outs = []
    for lo, hi in ((0, T1), (T1, 140)):
        T = hi - lo
        o = torch.empty((T, d.h_v, d.d_v), dtype=io, device="cuda")
        ws = torch.empty(gdn.gdn_prefill_workspace_size(d, T, 1), dtype=torch.uint8, device="cuda")
        gdn.gdn_prefill(d, cw, A, dt, dev(full["x"][lo:hi], io), dev(full["a"][lo:hi], io),
                        dev(full["b"][lo:hi], io), dev(np.array([0, T], np.int32)), slot, one,
                        state, conv, o, ws)
        outs.append(o)
    for t in range(140, 150):
        o = torch.empty((1, d.h_v, d.d_v), dtype=io, device="cuda")
        gdn.gdn_decode_step(d, cw, A, dt, dev(full["x"][t:t + 1], io), dev(full["a"][t:t + 1], io),
                            dev(full["b"][t:t + 1], io), slot, state, conv, o)
        outs.append(o)
    got = torch.cat(outs).float().cpu().numpy()
    from tests._gpu import assert_close_heads
    assert_close_heads(got, ref["o"], d, "o", head_axis=1)
    assert_close_heads(state[int(full["slot_idx"][0])].cpu().numpy(), ref["state"][0], d, "state",
                       head_axis=0)
    np.testing.assert_array_equal(conv[int(full["slot_idx"][0])].float().cpu().numpy(),
                                  ref["window"][0])


@pytest.mark.parametrize("name", sorted(SHAPES) + ["qwen35_4b_fp32_state"])
def test_prefill_with_empty_sequences_between(gpu_lib, name):
    """Empty sequences first, between and last: the chunk table of both
    prefill paths must map every chunk to the non-empty sequence it belongs
    to, and the empty sequences' slots get their initial state back."""
    d = (dataclasses.replace(QWEN35_4B, flags=gdn.GDN_FP32_STATE) if name.endswith("fp32_state")
         else SHAPES[name])
    lengths = [0, 17, 0, 0, 64, 1, 0, 130, 0]
    inp = workloads.layer_inputs(d, lengths, seed=zlib.crc32(name.encode()) % 10000, init="mixed",
                                 num_slots=len(lengths) + 2)
    run = PrefillRun(inp)
    run()
    check_prefill(inp, run.results(), oracle_prefill(inp, n_threads=NCPU))


@pytest.mark.parametrize("name", ["qwen35_4b", "tiny"])
def test_prefill_with_every_sequence_empty(gpu_lib, name):
    """No tokens at all (x, a, b and o empty): each sequence's slot gets its
    initial state and window back, or zeros without one; other slots stay bit
    for bit."""
    d = QWEN35_4B if name == "qwen35_4b" else TINY
    inp = workloads.layer_inputs(d, [0, 0, 0], seed=77, init="mixed", num_slots=5)
    run = PrefillRun(inp)
    run()
    check_prefill(inp, run.results(), oracle_prefill(inp))


def test_device_status_bits(gpu_lib):
    d = TINY
    inp = workloads.layer_inputs(d, [5, 7], seed=2, init="random", num_slots=4)
    # malformed cu_seqlens: nothing runs, status bit set, pools untouched
    bad = dict(inp, cu_seqlens=np.array([0, 9, 7], np.int32))
    run = PrefillRun(bad)
    run()
    g = run.results()
    assert g["status"] & gdn.GDN_DEV_BAD_CU_SEQLENS
    np.testing.assert_array_equal(g["state_pool"], inp["state_pool"])
    # out-of-range slot: that sequence is skipped, the other one runs
    bad2 = dict(inp, slot_idx=np.array([1, 99], np.int32))
    run = PrefillRun(bad2)
    run()
    g = run.results()
    assert g["status"] & gdn.GDN_DEV_BAD_SLOT
    ref = oracle_prefill(bad2 | {"slot_idx": np.array([1, 2], np.int32)})
    from tests._gpu import assert_close_heads
    assert_close_heads(g["state_pool"][1], ref["state"][0], d, "state seq 0", head_axis=0)
    # decode with an out-of-range slot
    dinp = workloads.decode_inputs(d, n_rows=3, num_slots=4, seed=1)
    dinp["slot_idx"] = np.array([0, 7, 2], np.int32)
    run = DecodeRun(dinp)
    run()
    g = run.results()
    assert g["status"] & gdn.GDN_DEV_BAD_SLOT
    assert not g["o"][1].any()


@pytest.mark.parametrize("dims", [TINY, QWEN35_4B], ids=["simt", "tensor_core"])
def test_prefill_negative_slot_sets_status_and_skips(gpu_lib, dims):
    """Prefill has no padding sequences: a negative slot is out of range like
    one past the pool, sets GDN_DEV_BAD_SLOT and leaves that sequence's o rows,
    and every slot, as they were; the other sequence runs normally."""
    inp = workloads.layer_inputs(dims, [70, 9], seed=12, init="random", num_slots=3)
    bad = dict(inp, slot_idx=np.array([-1, 2], np.int32))
    run = PrefillRun(bad)
    run()
    g = run.results()
    assert g["status"] & gdn.GDN_DEV_BAD_SLOT
    assert np.isnan(g["o"][:70]).all(), "the skipped sequence's o rows must not be written"
    for sl in (0, 1):
        np.testing.assert_array_equal(g["state_pool"][sl], inp["state_pool"][sl])
        np.testing.assert_array_equal(g["conv_pool"][sl], inp["conv_pool"][sl])
    ref = oracle_prefill(dict(bad, slot_idx=np.array([0, 2], np.int32)))
    from tests._gpu import assert_close_heads, assert_close_seq_out
    assert_close_seq_out(g["o"][70:], ref["o"][70:], dims, "o seq 1")
    assert_close_heads(g["state_pool"][2], ref["state"][1], dims, "state seq 1", head_axis=0)
    np.testing.assert_array_equal(g["conv_pool"][2], ref["window"][1].astype(np.float32))


# ---- full-size workloads, as the benchmark launches them ------------------

def test_qwen35_4b_prefill_full_size(gpu_lib):
    inp = workloads.prefill_4b()
    run = PrefillRun(inp)
    run()
    w = check_prefill(inp, run.results(), oracle_prefill(inp, n_threads=NCPU))
    print(f"prefill T=4096 worst normalised error {w:.3e}")


def test_decode_24_layers_64_slots_full_size_sampled(gpu_lib):
    """The 24 per-layer calls of one decode step (64 shuffled slots each), then
    every row of 3 sampled layers and 4 sampled rows of the rest against the
    oracle."""
    runs = [DecodeRun(workloads.decode_4b(layer)) for layer in range(24)]
    for r in runs:
        r()
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    full_layers = set(rng.choice(24, 3, replace=False).tolist())
    for layer, r in enumerate(runs):
        inp = r.inp
        rows = list(range(64)) if layer in full_layers else sorted(rng.choice(64, 4, replace=False))
        ref = oracle_decode(inp, rows=rows)
        g = r.results()
        sl = inp["slot_idx"]
        from tests._gpu import assert_close_rows
        assert_close_rows(g["o"][rows], ref["o"], inp["dims"], f"layer {layer} o row")
        assert_close_rows(g["state_pool"][sl[rows]], ref["state"], inp["dims"],
                          f"layer {layer} state row")
        np.testing.assert_array_equal(g["conv_pool"][sl[rows]], ref["window"].astype(np.float32))
        assert g["status"] == 0
