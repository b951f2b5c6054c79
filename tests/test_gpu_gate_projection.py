"""gdn_gate_projection: the decay and beta input projections as one matmul on
the tensor cores, against the float64 oracle (oracle.gate_projection).

Bound, per element: the kernel accumulates bf16 products in fp32 and rounds
once to bf16, so |err| <= 2^-8 |ref| (the final rounding, 2^-9, with margin)
+ 1e-3 max|ref| (the fp32 sum over d_model terms, orders of magnitude below
that).  A wrong weight row, a swapped a / b, a transposed operand or a lost K
block moves outputs by O(max|ref|) and fails it.

Shapes cover one and several K blocks per cluster rank (K split 1, 2 and 4,
even and uneven block counts), N = 2 h_v from 32 to 256 (16-column groups
on both sides of the a / b boundary), ragged token tails and a single token,
and the full 4B size
(T = 4096 tokens of width 2560).  The last test feeds the projected gates to
gdn_prefill and compares the layer with the oracle's projection and layer.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
import oracle
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B
from tests._gpu import PrefillRun, check_prefill, dev, oracle_prefill

pytestmark = pytest.mark.gpu


def _run(inp, dims):
    hidden = dev(inp["hidden"], torch.bfloat16)
    w = dev(inp["w_ba"], torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b = gdn.gdn_gate_projection(dims, hidden, w, d_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return a.float().cpu().numpy(), b.float().cpu().numpy()


def _check(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, what
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside the bound, worst "
                           f"{float((np.abs(got - ref) - bound).max()):.3e}")


@pytest.mark.parametrize("n,d_model,h_v", [
    (300, 256, 32),     # four K blocks: split 4, one block per rank; ragged tail of 44
    (128, 64, 16),      # one K block: no split; N = 32
    (200, 192, 48),     # three K blocks: split 2 (two and one); N = 96
    (1, 640, 128),      # one token, N = 256, ten blocks over four ranks
    (130, 320, 32),     # five blocks over four ranks (two, one, one, one)
    (257, 576, 16),     # nine blocks over four ranks (three, two, two, two)
    (4096, 2560, 32),   # the 4B size: 32 tiles x 40 K blocks
])
def test_gate_projection_matches_oracle(gpu_lib, n, d_model, h_v):
    inp = workloads.gate_projection_inputs(n, d_model, h_v, seed=1606 + n)
    dims = dataclasses.replace(QWEN35_4B, h_k=h_v // 2, h_v=h_v)
    a, b = _run(inp, dims)
    ra, rb = oracle.gate_projection(inp["hidden"], inp["w_ba"], h_v)
    _check(a, ra, f"a ({n}, {d_model}, {h_v})")
    _check(b, rb, f"b ({n}, {d_model}, {h_v})")


def test_gate_projection_rejects_before_launching(gpu_lib):
    inp = workloads.gate_projection_inputs(64, 128, 32)
    hidden = dev(inp["hidden"], torch.bfloat16)
    w = dev(inp["w_ba"], torch.bfloat16)
    a = torch.zeros((64, 32), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros_like(a)
    with pytest.raises(gdn.GdnError) as e:   # h_v = 2: not a multiple of 16
        gdn.gdn_gate_projection(workloads.TINY, hidden[:, :128], w[:4], a=a[:, :2].contiguous(),
                                b=b[:, :2].contiguous())
    assert e.value.status == -2   # GDN_EUNSUPPORTED
    with pytest.raises(gdn.GdnError) as e:   # d_model = 96: not a multiple of 64
        gdn.gdn_gate_projection(QWEN35_4B, hidden[:, :96].contiguous(), w[:, :96].contiguous(),
                                a=a, b=b)
    assert e.value.status == -2
    # n = 0 does nothing
    empty = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    a0, b0 = gdn.gdn_gate_projection(QWEN35_4B, empty, w)
    assert a0.shape == (0, 32) and b0.shape == (0, 32)
    torch.cuda.synchronize()
    assert not a.any() and not b.any()


def test_projected_gates_feed_the_prefill(gpu_lib):
    """hidden -> gdn_gate_projection -> gdn_prefill against the oracle's
    projection (rounded to bf16, the prefill's input type) and layer."""
    lengths = [130, 64, 7]
    inp = workloads.layer_inputs(QWEN35_4B, lengths, seed=1707, init="mixed")
    proj = workloads.gate_projection_inputs(sum(lengths), seed=1708)
    ra, rb = oracle.gate_projection(proj["hidden"], proj["w_ba"], QWEN35_4B.h_v)
    ref_inp = dict(inp, a=workloads.round_bf16(ra.astype(np.float32)),
                   b=workloads.round_bf16(rb.astype(np.float32)))
    run = PrefillRun(ref_inp)
    run.a, run.b = gdn.gdn_gate_projection(QWEN35_4B, dev(proj["hidden"], torch.bfloat16),
                                           dev(proj["w_ba"], torch.bfloat16))
    run()
    got = run.results()
    assert got["status"] == 0
    check_prefill(ref_inp, got, oracle_prefill(ref_inp))
