"""Which prefill path a call takes, read from the stage trace (launch count and
stages run) of gdn_prefill_traced: the Qwen3.5-4B shape runs on the tensor
cores (set-up, prep, scan: three launches, the prep and the scan in one
overlapped stage while the chains fit on half the SMs, as separate stages
otherwise), every other shape and GDN_FP32_STATE on the SIMT path (argument
check, front end, window write-back, chunk factors, scan: five launches).  A
silent fall-back of the headline shape to the slower path fails here."""
import dataclasses

import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, Dims
from tests._gpu import PrefillRun

pytestmark = pytest.mark.gpu


def _trace(d, lengths):
    inp = workloads.layer_inputs(d, lengths, seed=321)
    run = PrefillRun(inp)
    tr = gdn.make_trace()
    gdn.gdn_prefill(run.dims, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu, run.slot,
                    run.init, run.state, run.conv, run.o, run.ws, d_status=run.status, trace=tr)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    return tr.launches, tr.stages_run


def test_qwen35_4b_runs_on_the_tensor_cores_overlapped(gpu_lib):
    launches, stages = _trace(QWEN35_4B, [300, 77])
    assert launches == 3
    assert stages == 0b101          # set-up, then prep and scan together in stage 2


def test_qwen35_4b_many_chains_run_prep_then_scan(gpu_lib):
    # 3 sequences x 32 value heads = 96 chains > half the SMs: prep, then scan
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_seq = sms // (2 * QWEN35_4B.h_v) + 1
    launches, stages = _trace(QWEN35_4B, [70] * n_seq)
    assert launches == 3
    assert stages == 0b111


@pytest.mark.parametrize("variant", ["fp32_state", "chunk32", "small_heads"])
def test_other_shapes_run_on_the_simt_path(gpu_lib, variant):
    d = {"fp32_state": dataclasses.replace(QWEN35_4B, flags=gdn.GDN_FP32_STATE),
         "chunk32": dataclasses.replace(QWEN35_4B, chunk=32),
         "small_heads": Dims(h_k=2, h_v=4, d_k=64, d_v=64, chunk=64, io="bf16")}[variant]
    launches, stages = _trace(d, [130, 5])
    assert launches == 5
    assert stages == 0b111          # front end, chunk factors, scan
