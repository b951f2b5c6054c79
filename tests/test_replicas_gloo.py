"""Multi-process (N>1) host path on CPU: two gloo ranks, each running its own
replica of the tiny layer through the float64 oracle, then the benchmark's
aggregation (max-over-ranks job time, whole-job throughput).  The layer has
no cross-GPU exchange, so replicas must agree bit for bit and the only
collective is the timing reduction."""
import hashlib
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from gated_deltanet_linear_07_gb300 import workloads
        inp = workloads.tiny()
        d = inp["dims"]
        ov = workloads.oracle_view(inp)
        ref = oracle.layer(inp["x"], inp["a"], inp["b"], inp["conv_weight"], inp["A_log"],
                           inp["dt_bias"], inp["cu_seqlens"], d.h_k, d.h_v, d.d_k, d.d_v,
                           window0=ov["window0"], state0=ov["state0"], l2_eps=d.l2_eps)
        h = hashlib.sha256(np.ascontiguousarray(ref["o"]).tobytes() +
                           np.ascontiguousarray(ref["state"]).tobytes()).digest()
        digests = [None] * world
        dist.all_gather_object(digests, h)
        # each rank reports a different step time; the job time is the slowest
        ms = bench.max_over_ranks(dist, world, 1.0 + rank, torch.device("cpu"))
        T = inp["x"].shape[0]
        value = bench.replica_throughput(world, T, ms)
        q.put((rank, digests, ms, value, T))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_agree_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, digests, ms, value, T in res:
        assert digests[0] == digests[1], "replicas of the same seeded workload differ"
        assert ms == 2.0                    # max over ranks of (1.0, 2.0)
        assert value == pytest.approx(world * T / 2e-3)


def test_reference_arm_rank_nonzero_does_no_work(monkeypatch):
    """Under torchrun only rank 0 runs and prints the reference arm."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 0, 2

    def boom(*a, **k):
        raise AssertionError("rank 1 must not time the oracle")

    monkeypatch.setattr(bench, "oracle_prefill_time", boom)
    assert bench.run_reference(Args()) == 0
