"""The per-stage NaN/Inf probe (gdn_dims.flags |= GDN_CHECK_FINITE): on finite
inputs it raises no bit and leaves every result bit for bit unchanged (also
with empty sequences and a sequence whose slot is out of range, whose rows
nothing writes); a NaN or Inf put into one input raises the bit of the stage
where it first appears."""
import dataclasses

import numpy as np
import pytest

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, Dims
from tests._gpu import PrefillRun

pytestmark = pytest.mark.gpu

NONFINITE = (gdn.GDN_DEV_NONFINITE_FRONTEND | gdn.GDN_DEV_NONFINITE_CHUNK
             | gdn.GDN_DEV_NONFINITE_OUT)
SHAPES = {
    "qwen35_4b": QWEN35_4B,                                              # tensor-core path
    "qwen35_4b_fp32_state": dataclasses.replace(QWEN35_4B, flags=gdn.GDN_FP32_STATE),
    "asym_bf16": Dims(h_k=1, h_v=2, d_k=16, d_v=32, chunk=32, io="bf16"),
}


def _checked(d):
    return dataclasses.replace(d, flags=d.flags | gdn.GDN_CHECK_FINITE)


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_probe_is_silent_on_finite_inputs_and_changes_nothing(gpu_lib, name):
    d = SHAPES[name]
    lengths = [0, 70, 1, 0, 129]
    inp = workloads.layer_inputs(d, lengths, seed=81, init="mixed", num_slots=8)
    inp["slot_idx"] = inp["slot_idx"].copy()
    inp["slot_idx"][2] = 99                    # out of range: skipped, never written
    plain = PrefillRun(inp)
    plain()
    base = plain.results()
    run = PrefillRun(dict(inp, dims=_checked(d)))
    run()
    got = run.results()
    assert got["status"] & gdn.GDN_DEV_BAD_SLOT
    assert got["status"] & NONFINITE == 0, hex(got["status"])
    for k in ("o", "state_pool", "conv_pool"):
        np.testing.assert_array_equal(got[k], base[k])


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_inf_in_x_is_reported_from_the_front_end(gpu_lib, name):
    d = _checked(SHAPES[name])
    inp = workloads.layer_inputs(d, [100, 40], seed=82)
    inp["x"] = inp["x"].copy()
    inp["x"][57, 3] = np.inf                   # a query channel of key head 0
    run = PrefillRun(inp)
    run()
    st = run.results()["status"]
    assert st & gdn.GDN_DEV_NONFINITE_FRONTEND, hex(st)


def test_nan_gate_input_is_reported_from_the_chunk_stage_on_the_tensor_cores(gpu_lib):
    """On the tensor-core path the gates live in the chunk records, so a NaN in
    a shows up in the chunk stage with the front end's [Q; K] tiles finite; the
    SIMT path writes the gates in its front end."""
    for d, stage in ((QWEN35_4B, gdn.GDN_DEV_NONFINITE_CHUNK),
                     (SHAPES["qwen35_4b_fp32_state"], gdn.GDN_DEV_NONFINITE_FRONTEND)):
        inp = workloads.layer_inputs(_checked(d), [100, 40], seed=83)
        inp["a"] = inp["a"].copy()
        inp["a"][70, 5] = np.nan
        run = PrefillRun(inp)
        run()
        st = run.results()["status"]
        assert st & stage, (d, hex(st))
        if stage == gdn.GDN_DEV_NONFINITE_CHUNK:
            assert not st & gdn.GDN_DEV_NONFINITE_FRONTEND, hex(st)
