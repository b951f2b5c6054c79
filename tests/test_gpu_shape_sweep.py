"""GPU parity over a seeded sweep of layer shapes the fixed parity cases leave
out: value-to-key head ratios 1, 2, 4 and 8 (the repeat-interleaved key head
of value head h is h / (h_v / h_k)), unequal d_k and d_v, every chunk length,
both I/O types, random lengths (empty, single-token, ragged) and initial
states.  Each shape runs a varlen prefill and a decode step against the
float64 oracle with the tolerances of tests/_gpu.py.  The shapes are drawn
once from a fixed seed, so a failure names a reproducible case."""
import numpy as np
import pytest

from gated_deltanet_linear_07_gb300 import workloads
from gated_deltanet_linear_07_gb300.workloads import Dims
from tests._gpu import (DecodeRun, PrefillRun, check_decode, check_prefill, oracle_decode,
                        oracle_prefill)

pytestmark = pytest.mark.gpu


def _sweep(n=12, seed=20260):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        g = int(rng.choice([1, 2, 4, 8]))
        h_k = int(rng.choice([1, 2, 3])) if g < 8 else int(rng.choice([1, 2]))
        d_k = int(rng.choice([16, 32, 64]))
        d_v = int(rng.choice([16, 32, 64]))
        chunk = int(rng.choice([16, 32, 64, 128]))
        io = str(rng.choice(["fp32", "bf16"]))
        n_seq = int(rng.integers(2, 6))
        lengths = [int(x) for x in rng.choice([0, 1, 2, 3, 17, 63, 64, 65, 129, 200, 257], n_seq)]
        init = str(rng.choice(["zero", "mixed", "random"]))
        cases.append((f"s{i}-g{g}-hk{h_k}-dk{d_k}-dv{d_v}-c{chunk}-{io}",
                      Dims(h_k=h_k, h_v=g * h_k, d_k=d_k, d_v=d_v, chunk=chunk, io=io),
                      lengths, init, seed + i))
    return cases


CASES = _sweep()


@pytest.mark.parametrize("name,d,lengths,init,seed", CASES, ids=[c[0] for c in CASES])
def test_swept_shape_prefill_and_decode_match_oracle(gpu_lib, name, d, lengths, init, seed):
    inp = workloads.layer_inputs(d, lengths, seed=seed, init=init, num_slots=len(lengths) + 2)
    run = PrefillRun(inp)
    run()
    check_prefill(inp, run.results(), oracle_prefill(inp))
    dinp = workloads.decode_inputs(d, n_rows=6, num_slots=9, seed=seed + 1, padding_rows=1)
    drun = DecodeRun(dinp)
    drun()
    check_decode(dinp, drun.results(), oracle_decode(dinp))


def test_sweep_covers_every_ratio_chunk_and_io():
    """The drawn shapes include each head ratio, chunk length and I/O type."""
    gs = {c[1].h_v // c[1].h_k for c in CASES}
    chunks = {c[1].chunk for c in CASES}
    ios = {c[1].io for c in CASES}
    assert {4, 8} <= gs and {16, 128} <= chunks and ios == {"fp32", "bf16"}, (gs, chunks, ios)
