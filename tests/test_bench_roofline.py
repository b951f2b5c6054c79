"""Host logic of bench.py's roofline lines (no GPU): the FLOPs each prefill
stage is credited with, and the DRAM traffic each line takes from
profiles/ncu_traffic.json.  Traffic is per launch, so a launch of another
workload (4 x 32768, the varlen batch) must take its own record, never the
T=4096 one, and a record whose kernel sources have changed since the capture
must read as null."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B  # noqa: E402


def test_method_flops_per_token_head():
    # five C x C x d and three C x d x d contractions per chunk of C tokens,
    # 2 FLOP per multiply-add: (5 C^2 d + 3 C d^2) 2 / C per token
    C, d = 64, 128
    assert bench.alg_flops_per_token_head(C, d) == (5 * C * C * d + 3 * C * d * d) * 2 // C


def test_stage_flops_add_up_to_the_method():
    T = 4096
    stage = {"frontend": 0.01, "chunk": 0.05, "scan": 0.08}
    _, tf = bench.prefill_roofline(QWEN35_4B, T, stage, 1000.0, "test")
    total = sum(tf[k] * stage[k] * 1e9 for k in tf)       # TFLOP/s x ms -> FLOP
    want = bench.alg_flops_per_token_head(QWEN35_4B.chunk, QWEN35_4B.d_k) * T * QWEN35_4B.h_v
    assert total == pytest.approx(want, rel=1e-12)


def _record(monkeypatch, tmp_path, recs):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.json").write_text(json.dumps(recs))
    csrc = tmp_path / "gated_deltanet_linear_07_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("gdn_prefill_tc.cu", "gdn_tc.cuh", "gdn_common.cuh"):
        (csrc / f).write_text("// " + f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))


def test_each_workload_takes_its_own_traffic_record(monkeypatch, tmp_path):
    _record(monkeypatch, tmp_path, {})
    sha = bench.source_sha("prefill_chunk")
    assert bench.source_sha("prefill_chunk:adversarial_4x32768") == sha
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({
        "prefill_chunk": {"source_sha": sha, "dram_bytes_per_launch": 1},
        "prefill_overlap": {"source_sha": sha, "dram_bytes_per_launch": 2},
        "prefill_chunk:adversarial_4x32768": {"source_sha": sha, "dram_bytes_per_launch": 3},
    }))
    serial = {"frontend": 0.01, "chunk": 2.0, "scan": 0.8}      # prep then scan
    overlap = {"frontend": 0.01, "scan": 0.13}                  # prep beside the scan
    roof, _ = bench.prefill_roofline(QWEN35_4B, 131072, serial, 1000.0, "t",
                                     workload="adversarial_4x32768")
    assert roof["traffic"] == 3 and "prep_persistent" in roof["kernel"]
    roof, _ = bench.prefill_roofline(QWEN35_4B, 72196, serial, 1000.0, "t", workload="varlen_16")
    assert roof["traffic"] is None            # no record of that launch: null, not T=4096's
    roof, _ = bench.prefill_roofline(QWEN35_4B, 4096, overlap, 1000.0, "t")
    assert roof["traffic"] == 2
    roof, _ = bench.prefill_roofline(QWEN35_4B, 4096, serial, 1000.0, "t")
    assert roof["traffic"] == 1


def test_changed_sources_void_the_record(monkeypatch, tmp_path):
    _record(monkeypatch, tmp_path, {})
    sha = bench.source_sha("prefill_chunk")
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({
        "prefill_chunk:adversarial_4x32768": {"source_sha": sha, "dram_bytes_per_launch": 3}}))
    assert bench.recorded_traffic("prefill_chunk:adversarial_4x32768") == 3
    (tmp_path / "gated_deltanet_linear_07_gb300" / "csrc" / "gdn_prefill_tc.cu").write_text("// changed")
    assert bench.recorded_traffic("prefill_chunk:adversarial_4x32768") is None


def test_committed_records_name_their_summaries():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        recs = json.load(f)
    for key, rec in recs.items():
        assert rec["dram_bytes_per_launch"] > 0, key
        assert os.path.exists(os.path.join(ROOT, rec["summary"])), (key, rec["summary"])
        assert key.split(":")[0] in bench.KERNEL_SOURCES, key


def test_line_dtype_names_the_arithmetic_of_the_path_taken():
    import dataclasses
    from gated_deltanet_linear_07_gb300 import _binding as b
    from gated_deltanet_linear_07_gb300.workloads import TINY
    assert bench.prefill_dtype(QWEN35_4B) == "fp16"      # tensor-core default: fp16 operands
    assert bench.prefill_dtype(dataclasses.replace(QWEN35_4B, flags=b.GDN_BF16_OPERANDS)) == "bf16"
    assert bench.prefill_dtype(dataclasses.replace(QWEN35_4B, flags=b.GDN_FP32_STATE)) == "f32"
    assert bench.prefill_dtype(dataclasses.replace(QWEN35_4B, chunk=32)) == "f32"   # SIMT path
    assert bench.prefill_dtype(TINY) == "f32"
