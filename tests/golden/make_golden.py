"""Writes tests/golden/tiny_oracle.json from the float64 oracle (and nothing
else): a regression fixture of the tiny workload (1 sequence, T=64,
H_k=H_v=2, d_k=d_v=16, fp32, zero initial state), so that a rebuilt oracle on
another host (x86 here, Arm on the GPU host) is checked to reproduce it.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gated_deltanet_linear_07_gb300 import workloads  # noqa: E402


def compute():
    inp = workloads.tiny()
    d = inp["dims"]
    ov = workloads.oracle_view(inp)
    r = oracle.layer(inp["x"], inp["a"], inp["b"], inp["conv_weight"], inp["A_log"],
                     inp["dt_bias"], inp["cu_seqlens"], d.h_k, d.h_v, d.d_k, d.d_v,
                     window0=ov["window0"], state0=ov["state0"], n_threads=1)
    return {
        "o_tokens_0_3_63_head_1": [r["o"][t, 1].tolist() for t in (0, 3, 63)],
        "state_head_0_row_5": r["state"][0, 0, 5].tolist(),
        "o_abs_sum": float(abs(r["o"]).sum()),
        "state_abs_sum": float(abs(r["state"]).sum()),
    }


if __name__ == "__main__":
    out = {"what": "float64 oracle on the tiny workload (seed 1001); regression fixture",
           "written_by": "tests/golden/make_golden.py", **compute()}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)
