"""GPU parity of the gated RMSNorm of the layer output (gdn_gated_rmsnorm, called
through the C ABI) against the float64 oracle on the same seeded inputs, with
the stated tolerances of tests/_gpu.py; every supported d_v, both I/O types,
in place and out of place, a row of zeros, rows of very different scale and
gates far in both tails; and at the Qwen3.5-4B T=4096 output size."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_07_gb300 as gdn
import oracle
from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import QWEN35_4B, TINY, Dims
from tests._gpu import assert_close_rows, dev, io_dtype

pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny_fp32": TINY,
    "asym_fp32": Dims(h_k=2, h_v=4, d_k=32, d_v=64, chunk=16, io="fp32"),
    "asym2_bf16": Dims(h_k=1, h_v=2, d_k=16, d_v=32, chunk=32, io="bf16"),
    "tall_fp32": Dims(h_k=1, h_v=1, d_k=128, d_v=16, chunk=64, io="fp32"),
    "qwen35_4b": QWEN35_4B,
}


def _inputs(d, n, seed):
    rng = np.random.default_rng(seed)
    o = rng.standard_normal((n, d.h_v, d.d_v)).astype(np.float32)
    o[0] = 0.0                                      # a zero row: y = 0
    if n > 2:
        o[1] *= 1e-3                                 # rows of very different scale
        o[2] *= 1e2
    z = (2.0 * rng.standard_normal((n, d.h_v, d.d_v))).astype(np.float32)
    z[-1, :, : d.d_v // 2] = 30.0                    # open gate
    z[-1, :, d.d_v // 2:] = -30.0                    # closed gate
    w = rng.uniform(0.25, 2.0, d.d_v).astype(np.float32)
    if d.io == "bf16":
        o, z = workloads.round_bf16(o), workloads.round_bf16(z)
    return o, z, w


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("in_place", [False, True])
def test_gated_rmsnorm_matches_oracle(gpu_lib, name, in_place):
    d = SHAPES[name]
    n = 37
    o, z, w = _inputs(d, n, seed=len(name) * 7 + in_place)
    io = io_dtype(d)
    do, dz, dw = dev(o, io), dev(z, io), dev(w)
    dy = do if in_place else torch.full_like(do, float("nan"))
    gdn.gdn_gated_rmsnorm(d, dw, do, dz, y=dy, eps=1e-6)
    torch.cuda.synchronize()
    got = dy.float().cpu().numpy()
    ref = oracle.gated_rmsnorm(o, z, w, eps=1e-6)
    assert_close_rows(got, ref, d, f"{name} y row")
    assert not got[0].any()
    if not in_place:   # the inputs are not touched
        np.testing.assert_array_equal(do.float().cpu().numpy(), o)


def test_gated_rmsnorm_qwen35_4b_full_output(gpu_lib):
    """The T=4096 x 32-head output of the Qwen3.5-4B layer, every row."""
    d = QWEN35_4B
    o, z, w = _inputs(d, 4096, seed=5)
    do, dz, dw = dev(o, torch.bfloat16), dev(z, torch.bfloat16), dev(w)
    dy = torch.empty_like(do)
    gdn.gdn_gated_rmsnorm(d, dw, do, dz, y=dy)
    torch.cuda.synchronize()
    got = dy.float().cpu().numpy()
    ref = oracle.gated_rmsnorm(o, z, w)
    worst = assert_close_rows(got, ref, d, "y row")
    # per row the result is only bf16 rounding away from the float64 one
    rows = np.abs(ref).max(axis=-1, keepdims=True) + 1e-30
    assert np.percentile(np.abs(got - ref) / rows, 99.9) < 1e-2
    print(f"gated norm T=4096 worst normalised error {worst:.3e}")
