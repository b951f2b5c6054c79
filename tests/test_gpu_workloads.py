"""Full-size workloads against the oracle on sampled (sequence, head) pairs.

- adversarial: 4 sequences x 32768 tokens, Qwen3.5-4B layer shape, random
  initial states and windows, key channels alternating 512-token runs of one
  repeated vector (fully correlated keys) with random segments, beta near 1;
  sub-case "b" also pins the decay near 1 (a = -12).  The oracle runs the
  token-by-token recurrence over the whole sequence for the sampled heads.
- varlen: 16 sequences with lengths ~ U{1..8192}, prefill through cu_seqlens,
  then 256 decode steps per sequence; one oracle recurrence over
  length + 256 tokens per sampled (sequence, head).
"""
import os

import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
import oracle
from gated_deltanet_linear_07_gb300 import workloads
from tests._gpu import PrefillRun, assert_close, dev, io_dtype

pytestmark = pytest.mark.gpu
NCPU = os.cpu_count() or 1


def _sample_mask(B, h_v, per_seq, seed):
    rng = np.random.default_rng(seed)
    mask = np.zeros((B, h_v), bool)
    for s in range(B):
        mask[s, rng.choice(h_v, per_seq, replace=False)] = True
    return mask


@pytest.mark.parametrize("sub", ["a", "b"])
def test_adversarial_long_prefill_sampled(gpu_lib, sub):
    inp = workloads.adversarial(sub=sub)
    d = inp["dims"]
    run = PrefillRun(inp)
    run()
    got = run.results()
    assert got["status"] == 0
    assert np.isfinite(got["o"]).all() and np.isfinite(got["state_pool"]).all()
    mask = _sample_mask(4, d.h_v, 2, seed=11)
    ov = workloads.oracle_view(inp)
    ref = oracle.layer(inp["x"], inp["a"], inp["b"], inp["conv_weight"], inp["A_log"],
                       inp["dt_bias"], inp["cu_seqlens"], d.h_k, d.h_v, d.d_k, d.d_v,
                       window0=ov["window0"], state0=ov["state0"], head_mask=mask,
                       n_threads=NCPU)
    cu = inp["cu_seqlens"]
    for s in range(4):
        slot = inp["slot_idx"][s]
        np.testing.assert_array_equal(got["conv_pool"][slot], ref["window"][s].astype(np.float32))
        for h in np.nonzero(mask[s])[0]:
            w = assert_close(got["o"][cu[s]:cu[s + 1], h], ref["o"][cu[s]:cu[s + 1], h], d,
                             f"o seq {s} head {h}")
            w2 = assert_close(got["state_pool"][slot, h], ref["state"][s, h], d,
                              f"state seq {s} head {h}")
            print(f"seq {s} head {h}: worst normalised error o {w:.2e} state {w2:.2e}")


def test_varlen_prefill_then_256_decode_steps_sampled(gpu_lib):
    inp = workloads.varlen()
    d = inp["dims"]
    io = io_dtype(d)
    B = len(inp["lengths"])
    run = PrefillRun(inp)
    run()
    pre = run.results()
    assert pre["status"] == 0
    steps = inp["decode_x"].shape[0]
    outs = []
    for t in range(steps):
        o = torch.empty((B, d.h_v, d.d_v), dtype=io, device="cuda")
        gdn.gdn_decode_step(d, run.cw, run.A_log, run.dt_bias, dev(inp["decode_x"][t], io),
                            dev(inp["decode_a"][t], io), dev(inp["decode_b"][t], io), run.slot,
                            run.state, run.conv, o, d_status=run.status)
        outs.append(o)
    dec = torch.stack(outs).float().cpu().numpy()          # [steps, B, h_v, d_v]
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    state = run.state.cpu().numpy()
    conv = run.conv.float().cpu().numpy()
    # one oracle recurrence over prefill + decode tokens per sequence
    cu = inp["cu_seqlens"]
    xs, as_, bs, lens = [], [], [], []
    for s in range(B):
        xs += [inp["x"][cu[s]:cu[s + 1]], inp["decode_x"][:, s]]
        as_ += [inp["a"][cu[s]:cu[s + 1]], inp["decode_a"][:, s]]
        bs += [inp["b"][cu[s]:cu[s + 1]], inp["decode_b"][:, s]]
        lens.append(int(cu[s + 1] - cu[s]) + steps)
    cu2 = np.concatenate([[0], np.cumsum(lens)])
    mask = _sample_mask(B, d.h_v, 3, seed=5)
    ref = oracle.layer(np.concatenate(xs), np.concatenate(as_), np.concatenate(bs),
                       inp["conv_weight"], inp["A_log"], inp["dt_bias"], cu2, d.h_k, d.h_v,
                       d.d_k, d.d_v, head_mask=mask, n_threads=NCPU)
    for s in range(B):
        slot = inp["slot_idx"][s]
        T = int(cu[s + 1] - cu[s])
        np.testing.assert_array_equal(conv[slot], ref["window"][s].astype(np.float32))
        for h in np.nonzero(mask[s])[0]:
            r = ref["o"][cu2[s]:cu2[s + 1], h]
            assert_close(pre["o"][cu[s]:cu[s + 1], h], r[:T], d, f"prefill o seq {s} head {h}")
            assert_close(dec[:, s, h], r[T:], d, f"decode o seq {s} head {h}")
            assert_close(state[slot, h], ref["state"][s, h], d, f"state seq {s} head {h}")
