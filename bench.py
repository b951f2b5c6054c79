#!/usr/bin/env python3
"""Benchmark of the Gated DeltaNet layer library on GB300.

One step = one gdn_prefill call over the Qwen3.5-4B-shaped layer workload
(B=1, T=4096, H_k=16 -> H_v=32, d_k=d_v=128, conv over 8192 channels, bf16
I/O, fp32 state, chunk 64, zero initial state), inputs resident in HBM, L2
flushed before every timed step (a 256 MiB write, then a 256 MiB read so the
write-backs land outside the timed region).  The same JSON line also
carries the decode step (24 layers x 64 slots, one bf16 token per slot,
shuffled slots, random fp32 states) as a second measured quantity, the
large prefill workloads (4 x 32768 adversarial, a 16-sequence varlen batch)
with their rooflines, the end-to-end figure through the C ABI with host
buffers (and the host link's plain-copy ceiling), the side operations (gated
norm, decay/beta projection, slot copy, checkpointed and fp32-state
prefills), side figures outside the headline (the prefill with a warm L2;
the prefill and the decode step replayed from CUDA graphs), the roofline of
the dominant kernel and the float64 CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

With N > 1 it is launched by torch.distributed.run, one rank per GPU; every
rank runs its own replica of the workload (the layer has no cross-GPU
exchange) and rank 0 prints the line with the max-over-ranks time.
--impl reference times the float64 CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s (%TC roofline); decode state GB/s (%HBM peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("gdn", "reference"), default="gdn")
    p.add_argument("--decode-steps", type=int, default=None,
                   help="timed decode steps (default: --steps)")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-prefill", action="store_true",
                   help="measure only the decode step (profiling runs)")
    p.add_argument("--decode-layers", type=int, default=24)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the warm-L2 and CUDA-graph side figures")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-large", action="store_true",
                   help="skip the 4 x 32768 and the mixed varlen prefill workloads")
    p.add_argument("--large-only", action="store_true",
                   help="only the 4 x 32768 and the mixed varlen prefill workloads")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        loaded = [v for v in sm if mx and v >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


def gpu_id_of(torch, dev_index):
    try:
        props = torch.cuda.get_device_properties(dev_index)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", None)
        pdev = getattr(props, "pci_device_id", None)
        if bus is not None and dom is not None and pdev is not None:
            return f"{dom:08x}:{bus:02x}:{pdev:02x}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev_index]
    return str(dev_index)


# ---------------------------------------------------------------- workloads

class L2Flush:
    """Before a timed call: write a buffer larger than L2 (evicting the
    inputs), then read another one, so the write's dirty lines are written
    back before the timed region instead of inside it."""

    def __init__(self, torch, device):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty(1, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.fill_(1.0)
        self.sink.copy_(self.r.sum().reshape(1))


def alg_flops_per_token_head(C, d):
    """Method FLOPs per (token, value head): five C x C x d contractions
    (K K^T, Q K^T, T (beta V), T (beta e^gamma K), P W) and three C x d x d
    contractions (Wk S^T, Q S^T, W^T K) per chunk, 2 FLOP per multiply-add."""
    return 10 * C * d + 6 * d * d


KERNEL_SOURCES = {
    "decode_step": ("gdn_decode.cu", "gdn_common.cuh"),
    "prefill_scan": ("gdn_prefill_tc.cu", "gdn_tc.cuh", "gdn_common.cuh"),
    "prefill_chunk": ("gdn_prefill_tc.cu", "gdn_tc.cuh", "gdn_common.cuh"),
    "prefill_overlap": ("gdn_prefill_tc.cu", "gdn_tc.cuh", "gdn_common.cuh"),
    "gated_norm": ("gdn_norm.cu", "gdn_common.cuh"),
    "slot_copy": ("gdn_slots.cu", "gdn_common.cuh"),
    "gate_projection": ("gdn_proj.cu", "gdn_tc.cuh", "gdn_common.cuh"),
}


def source_sha(kernel_key):
    """Hash of the sources a kernel is built from (the files named in
    KERNEL_SOURCES; all of csrc/ for a kernel not listed).  A key of the form
    'kernel:workload' takes the kernel's sources."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_linear_07_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel_key.split(":")[0]) or sorted(
        f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh")))
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch of a kernel from the committed ncu summary, if its
    sources have not changed since the counters were taken.  The key names the
    kernel and, after a colon, the workload when the launch is not the T=4096
    one (traffic is per launch, so each workload has its own record)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_key)
    if not rec or rec.get("source_sha") != source_sha(kernel_key):
        return None
    return rec.get("dram_bytes_per_launch")


class Prefill:
    def __init__(self, torch, gdn, inp, device):
        d = inp["dims"]
        self.torch, self.gdn, self.inp, self.dims = torch, gdn, inp, d
        io = torch.bfloat16 if d.io == "bf16" else torch.float32
        self.io = io
        t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)  # noqa: E731
        self.host = {k: inp[k] for k in ("x", "a", "b")}
        self.x, self.a, self.b = t(inp["x"], io), t(inp["a"], io), t(inp["b"], io)
        self.cw, self.A_log, self.dt_bias = t(inp["conv_weight"]), t(inp["A_log"]), t(inp["dt_bias"])
        self.cu = t(inp["cu_seqlens"].astype(np.int32))
        self.slot = t(inp["slot_idx"].astype(np.int32))
        self.init = t(inp["has_init"].astype(np.uint8))
        self.state = t(inp["state_pool"])
        self.conv = t(inp["conv_pool"], io)
        T = inp["x"].shape[0]
        self.T = T
        self.o = torch.empty((T, d.h_v, d.d_v), dtype=io, device=device)
        ws = gdn.gdn_prefill_workspace_size(d, T, len(inp["lengths"]))
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def __call__(self, trace=None, x=None, a=None, b=None, cu=None, slot=None, init=None, o=None):
        self.gdn.gdn_prefill(self.dims, self.cw, self.A_log, self.dt_bias,
                             self.x if x is None else x, self.a if a is None else a,
                             self.b if b is None else b, self.cu if cu is None else cu,
                             self.slot if slot is None else slot, self.init if init is None else init,
                             self.state, self.conv, self.o if o is None else o, self.ws,
                             d_status=self.status, trace=trace)


class DevicePrefill(Prefill):
    """A prefill workload whose inputs were drawn on the device
    (device_layer_inputs); the call is Prefill's."""

    def __init__(self, torch, gdn, dinp, device):
        d = dinp["dims"]
        self.torch, self.gdn, self.inp, self.dims = torch, gdn, dinp, d
        self.io = torch.bfloat16 if d.io == "bf16" else torch.float32
        self.host = None
        for k in ("x", "a", "b", "cw", "A_log", "dt_bias", "cu", "slot", "init", "state", "conv"):
            setattr(self, k, dinp[k])
        T = dinp["x"].shape[0]
        self.T = T
        self.o = torch.empty((T, d.h_v, d.d_v), dtype=self.io, device=device)
        ws = gdn.gdn_prefill_workspace_size(d, T, len(dinp["lengths"]))
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)


def device_layer_inputs(torch, device, dims, lengths, seed, *, init="zero", b_mean=0.0,
                        a_const=None, correlated_keys=0, state_std=0.02):
    """The recipe of workloads.layer_inputs (same distributions and structure:
    x, a, b ~ N(0, 1), b shifted by b_mean, a optionally constant, conv weight
    ~ N(0, 0.5^2), A_log ~ U(0, 2.7), dt_bias ~ N(0, 0.1^2), states ~
    N(0, state_std^2), windows ~ N(0, 1), shuffled slots, key channels of x in
    alternating runs of one repeated vector and random segments) drawn on the
    device with a seeded torch generator.  The large benchmark workloads take
    minutes to draw on the host; these are timed, not compared with the
    oracle (the parity tests draw theirs on the host)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    io = torch.bfloat16 if dims.io == "bf16" else torch.float32
    B = len(lengths)
    cu = np.zeros(B + 1, np.int64)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    randn = lambda *shape: torch.randn(*shape, generator=g, device=device)  # noqa: E731
    x = randn(T, dims.conv_dim)
    if correlated_keys:
        R = int(correlated_keys)
        k0, k1 = dims.h_k * dims.d_k, 2 * dims.h_k * dims.d_k
        for s in range(B):
            for r0 in range(0, int(lengths[s]), 2 * R):
                r1 = min(r0 + R, int(lengths[s]))
                x[int(cu[s]) + r0:int(cu[s]) + r1, k0:k1] = randn(1, k1 - k0)
    a = randn(T, dims.h_v)
    if a_const is not None:
        a.fill_(a_const)
    b = randn(T, dims.h_v) + b_mean
    num_slots = B
    perm = torch.randperm(num_slots, generator=g, device=device)
    has_init = torch.full((B,), 1 if init == "random" else 0, dtype=torch.uint8, device=device)
    return {
        "dims": dims, "lengths": [int(t) for t in lengths],
        "x": x.to(io), "a": a.to(io), "b": b.to(io),
        "cw": randn(dims.conv_dim, dims.conv_w) * 0.5,
        "A_log": torch.rand(dims.h_v, generator=g, device=device) * 2.7,
        "dt_bias": randn(dims.h_v) * 0.1,
        "cu": torch.from_numpy(cu.astype(np.int32)).to(device),
        "slot": perm[:B].to(torch.int32).contiguous(), "init": has_init,
        "state": randn(num_slots, dims.h_v, dims.d_k, dims.d_v) * state_std,
        "conv": randn(num_slots, dims.conv_w - 1, dims.conv_dim).to(io),
    }


def trace_stages(torch, gdn, run, ev, flush):
    """Attribution pass: the steps again with stage events and a launch count
    (the events sit between kernels, so this pass is not the headline).
    Returns the median ms of each stage that ran and the launches counted."""
    launches = 0
    traces = []
    for e in ev:
        flush()
        tr = gdn.make_trace(e["b"], e["f"])
        run(trace=tr)
        launches += tr.launches
        traces.append(tr)
    torch.cuda.synchronize()
    stage_ms = {}
    for i, name in enumerate(gdn.STAGES):
        vals = [e["b"][i].elapsed_time(e["f"][i]) for e, tr in zip(ev, traces)
                if tr.stages_run & (1 << i)]
        if vals:
            stage_ms[name] = statistics.median(vals)
    return stage_ms, launches


def graph_replay_ms(torch, fn, steps, flush=None):
    """`fn` (library calls on the current stream) captured once into a CUDA
    graph and replayed: the median ms of `steps` replays with CUDA events
    around each, `flush` (outside the graph) before each when given.  Returns
    (ms, None), or (None, reason) when the capture is refused."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        # thread-local: only this thread's calls are checked during the capture
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
    except RuntimeError as e:
        torch.cuda.synchronize()
        return None, (str(e).strip().splitlines() or ["capture failed"])[0][:200]
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(steps)]
    for s_, e_ in ev:
        if flush is not None:
            flush()
        s_.record()
        g.replay()
        e_.record()
    torch.cuda.synchronize()
    ms = statistics.median(s_.elapsed_time(e_) for s_, e_ in ev)
    del g
    return ms, None


def warm_l2_ms(torch, fn, steps):
    """Median ms of `fn` called back to back without an L2 flush (inputs that
    fit in L2 stay there), CUDA events around each call."""
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for _ in range(3):
        fn()
    ev = [(mk(), mk()) for _ in range(steps)]
    for s_, e_ in ev:
        s_.record()
        fn()
        e_.record()
    torch.cuda.synchronize()
    return statistics.median(s_.elapsed_time(e_) for s_, e_ in ev)


def bench_launch_variants(torch, pf_run, steps, device):
    """Side figures of the T=4096 prefill outside the headline: back to back
    with a warm L2, and replayed from a CUDA graph (L2 flushed before each)."""
    out = {"prefill_warm_l2_ms": warm_l2_ms(torch, pf_run, steps)}
    ms, why = graph_replay_ms(torch, pf_run, steps, flush=L2Flush(torch, device))
    out["prefill_cuda_graph_ms"] = ms
    if why:
        out["prefill_cuda_graph_error"] = why
    out["note"] = ("not the headline: warm = no L2 flush between calls; graph = the same call "
                   "captured once with torch.cuda.CUDAGraph and replayed")
    return out


def bench_prefill(torch, gdn, workloads, device, steps, warmup):
    inp = workloads.prefill_4b()
    run = Prefill(torch, gdn, inp, device)
    out = time_prefill(torch, gdn, run, L2Flush(torch, device), steps, warmup)
    out["inp"] = inp
    return out


def time_prefill(torch, gdn, run, flush, steps, warmup):
    """K timed calls of `run` (L2 flushed before each), then the stage
    attribution pass."""
    ns = gdn.STAGES
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for _ in range(max(warmup, 1)):
        run()
    torch.cuda.synchronize()
    ev = [{"s": mk(), "e": mk(), "b": [mk() for _ in ns], "f": [mk() for _ in ns]}
          for _ in range(steps)]
    stream = torch.cuda.current_stream()
    for e in ev:   # create the event handles before handing them to the library
        for x in [e["s"], e["e"], *e["b"], *e["f"]]:
            x.record(stream)
    torch.cuda.synchronize()
    # Timed pass: the plain call, events only around each step.
    for e in ev:
        flush()
        e["s"].record(stream)
        run()
        e["e"].record(stream)
    torch.cuda.synchronize()
    step_ms = [e["s"].elapsed_time(e["e"]) for e in ev]
    stage_ms, launches = trace_stages(torch, gdn, run, ev, flush)
    status = int(run.status.item())
    return {"run": run, "step_ms": step_ms, "stage_ms": stage_ms,
            "launches": launches, "status": status}


LARGE_WORKLOADS = {
    "adversarial_4x32768": "4 sequences x 32768 tokens of the Qwen3.5-4B layer, bf16, random "
                           "initial states and windows, key channels in alternating 512-token "
                           "runs of one repeated vector and random segments, b ~ N(6, 1)",
    "varlen_16": "16 sequences of U{1..8192} tokens (cu_seqlens) of the Qwen3.5-4B layer, bf16, "
                 "zero initial state, shuffled slots; then 256 decode steps per sequence",
}


def bench_large(torch, gdn, workloads, device, name, steps, warmup, peak_tf, peak_src, hbm):
    """One of the large prefill workloads: K timed calls (L2 flushed before
    each; the inputs are larger than L2 as well), the stage split, the
    roofline of the dominant stage and the whole-call fraction; for the
    varlen batch also its 256 decode steps."""
    d = workloads.QWEN35_4B
    if name == "adversarial_4x32768":
        lengths = [32768] * 4
        dinp = device_layer_inputs(torch, device, d, lengths, workloads.SEED_BASE + 4,
                                   init="random", b_mean=6.0, correlated_keys=512)
    else:
        lengths, _ = workloads.varlen_lengths()
        dinp = device_layer_inputs(torch, device, d, lengths.tolist(), workloads.SEED_BASE + 5)
    run = DevicePrefill(torch, gdn, dinp, device)
    res = time_prefill(torch, gdn, run, L2Flush(torch, device), steps, warmup)
    T = run.T
    ms = statistics.median(res["step_ms"])
    roof, stage_tflops = prefill_roofline(d, T, res["stage_ms"], peak_tf, peak_src, workload=name)
    flops = alg_flops_per_token_head(d.chunk, d.d_k) * T * d.h_v
    # minimum HBM bytes of the call: x, a, b in, o out, initial states read, final written
    nb = len(lengths)
    state_b = d.h_v * d.d_k * d.d_v * 4
    min_bytes = T * (d.conv_dim * 2 + 2 * d.h_v * 2 + d.h_v * d.d_v * 2) + \
        nb * state_b * (2 if name == "adversarial_4x32768" else 1)
    out = {"metric": "GDN prefill tokens/s", "value": T / (ms / 1e3), "unit": "tokens/s",
           "ms_per_step": ms, "steps": steps,
           "config": {"workload": LARGE_WORKLOADS[name], "B": nb, "T": T, "chunk": d.chunk,
                      "io": d.io, "data": "synthetic, drawn on the device (seeded)",
                      "l2": "flushed before every timed step; inputs larger than L2"},
           "roofline": roof, "stages_ms": res["stage_ms"], "stages_tflops": stage_tflops,
           "tc_roofline_frac_whole_step": flops / (ms / 1e3) / 1e12 / peak_tf,
           "flops_per_step": flops, "min_hbm_bytes_per_step": min_bytes,
           "hbm_floor_frac_of_tc_roofline": (flops / peak_tf / 1e12) /
                                            (min_bytes / hbm / 1e9),
           "gpu_launches": res["launches"], "device_status": res["status"]}
    if name == "varlen_16":
        out["decode_after_prefill"] = bench_varlen_decode(torch, gdn, run, steps, warmup)
    del run, dinp
    torch.cuda.empty_cache()
    return out


def bench_varlen_decode(torch, gdn, run, steps, warmup, n_steps=256):
    """The varlen batch's 256 decode steps after its prefill: one token per
    sequence per step on the slots the prefill wrote, back to back."""
    d = run.dims
    B = len(run.inp["lengths"])
    g = torch.Generator(device=run.x.device)
    g.manual_seed(5005)
    xs = torch.randn(n_steps, B, d.conv_dim, generator=g, device=run.x.device).to(run.io)
    abs_ = torch.randn(2, n_steps, B, d.h_v, generator=g, device=run.x.device).to(run.io)
    o = torch.empty((B, d.h_v, d.d_v), dtype=run.io, device=run.x.device)
    status = torch.zeros(1, dtype=torch.int32, device=run.x.device)

    def all_steps():
        for t in range(n_steps):
            gdn.gdn_decode_step(d, run.cw, run.A_log, run.dt_bias, xs[t], abs_[0, t], abs_[1, t],
                                run.slot, run.state, run.conv, o, d_status=status)
    for _ in range(max(warmup, 1)):
        all_steps()
    torch.cuda.synchronize()
    times = []
    for _ in range(max(steps // 4, 3)):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        all_steps()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) / n_steps)
    ms = statistics.median(times)
    sb = B * 2 * d.h_v * d.d_k * d.d_v * 4
    return {"metric": "decode state GB/s", "value": sb / (ms / 1e3) / 1e9, "unit": "GB/s",
            "ms_per_step": ms, "rows_per_step": B, "state_bytes_per_step": sb,
            "note": "16 slots of state (64 MiB) stay resident in L2 across the back-to-back "
                    "steps, so this is not an HBM roofline figure",
            "device_status": int(status.item())}


def bench_e2e(torch, gdn, run, steps, warmup):
    """Host (pinned) inputs -> H2D -> gdn_prefill -> D2H of the output, every
    step inside the timed region, pipelined the way a serving loop runs it:
    two device buffer sets, the uploads on one stream, the layer on another,
    the downloads on a third, so that step i's compute overlaps step i+1's
    upload and step i-1's download.  Steps are ordered through the buffers'
    events only; the layer calls themselves run one after another."""
    inp = run.inp
    io = run.io
    pin = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a)).to(dtype=dt).pin_memory()  # noqa: E731
    host_in = (pin(inp["x"], io), pin(inp["a"], io), pin(inp["b"], io),
               pin(inp["cu_seqlens"].astype(np.int32)), pin(inp["slot_idx"].astype(np.int32)),
               pin(inp["has_init"].astype(np.uint8)))
    dev = run.x.device
    nbuf = 2
    dev_in = [tuple(torch.empty_like(t, device=dev) for t in host_in) for _ in range(nbuf)]
    dev_out = [torch.empty(run.o.shape, dtype=io, device=dev) for _ in range(nbuf)]
    host_out = [torch.empty(run.o.shape, dtype=io).pin_memory() for _ in range(nbuf)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]    # buffer k's inputs have landed
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]   # the layer on buffer k is done
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]   # buffer k's output is on the host
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()

    def step(i):
        k = i % nbuf
        s_in.wait_event(ev_cmp[k])              # the layer that read buffer k is done
        with torch.cuda.stream(s_in):
            for d_, h_ in zip(dev_in[k], host_in):
                d_.copy_(h_, non_blocking=True)
        ev_in[k].record(s_in)
        s_cmp.wait_event(ev_in[k])
        s_cmp.wait_event(ev_out[k])             # buffer k's previous output has been read
        with torch.cuda.stream(s_cmp):
            dx, da, db, dcu, dslot, dinit = dev_in[k]
            run(x=dx, a=da, b=db, cu=dcu, slot=dslot, init=dinit, o=dev_out[k])
        ev_cmp[k].record(s_cmp)
        s_out.wait_event(ev_cmp[k])
        with torch.cuda.stream(s_out):
            host_out[k].copy_(dev_out[k], non_blocking=True)
        ev_out[k].record(s_out)

    for i in range(max(warmup, 1)):
        step(i)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(s_in)
    for i in range(steps):
        step(i)
    e.record(s_out)                             # after the last download
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    # the last step's output arrived intact
    np.testing.assert_array_equal(host_out[(steps - 1) % nbuf].float().numpy(),
                                  dev_out[(steps - 1) % nbuf].float().cpu().numpy())
    # What the host link gives one plain copy of the same size, each direction alone
    # (pinned memory, one cudaMemcpyAsync): the ceiling the pipeline is held to.
    def link(dst, src):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(5):
            t0.record()
            dst.copy_(src, non_blocking=True)
            t1.record()
            torch.cuda.synchronize()
            ts.append(t0.elapsed_time(t1))
        return dst.numel() * dst.element_size() / (statistics.median(ts) / 1e3) / 1e9
    h2d_gbs = link(dev_in[0][0], host_in[0])
    d2h_gbs = link(host_out[0], dev_out[0])
    return {"ms": ms, "h2d": h2d, "d2h": d2h, "pipeline": f"{nbuf} buffer sets, 3 streams",
            "link": {"h2d_gbs_plain_copy": h2d_gbs, "d2h_gbs_plain_copy": d2h_gbs,
                     "what": "one pinned copy of x (H2D) and of o (D2H), each alone"}}


def bench_gated_norm(torch, gdn, dims, T, device, steps, warmup):
    """Gated RMSNorm of a T-token layer output (o, z [T, h_v, d_v] in the I/O
    dtype, out of place), L2 flushed before every timed call."""
    io = torch.bfloat16 if dims.io == "bf16" else torch.float32
    g = torch.Generator(device=device).manual_seed(1234)
    o = torch.randn((T, dims.h_v, dims.d_v), generator=g, device=device).to(io)
    z = torch.randn((T, dims.h_v, dims.d_v), generator=g, device=device).to(io)
    w = torch.rand(dims.d_v, generator=g, device=device) + 0.5
    y = torch.empty_like(o)
    flush = L2Flush(torch, device)
    for _ in range(max(warmup, 1)):
        gdn.gdn_gated_rmsnorm(dims, w, o, z, y=y)
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(steps)]
    for a_, b_ in ev:
        flush()
        a_.record()
        gdn.gdn_gated_rmsnorm(dims, w, o, z, y=y)
        b_.record()
    torch.cuda.synchronize()
    ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in ev)
    nbytes = 3 * o.numel() * o.element_size()
    return {"ms": ms, "bytes": nbytes, "rows": T * dims.h_v}


def bench_gate_projection(torch, gdn, workloads, dims, T, device, steps, warmup):
    """The decay and beta input projections of a T-token batch as one launch
    (gdn_gate_projection: hidden [T, 2560] bf16, both weights in one [2 h_v,
    2560] matrix), and the same two products as two separate library matmuls
    (cuBLAS through torch) for comparison; L2 flushed before every timed call."""
    inp = workloads.gate_projection_inputs(T, h_v=dims.h_v)
    bf = torch.bfloat16
    hidden = torch.from_numpy(inp["hidden"]).to(device=device, dtype=bf)
    w = torch.from_numpy(inp["w_ba"]).to(device=device, dtype=bf)
    h_v = dims.h_v
    a = torch.empty((T, h_v), dtype=bf, device=device)
    b = torch.empty_like(a)
    a2, b2 = torch.empty_like(a), torch.empty_like(a)
    w_a, w_b = w[:h_v].t(), w[h_v:].t()
    flush = L2Flush(torch, device)
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def timed(fn):
        for _ in range(max(warmup, 3)):
            fn()
        ev = [(mk(), mk()) for _ in range(steps)]
        for e0, e1 in ev:
            flush()
            e0.record()
            fn()
            e1.record()
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)

    status = torch.zeros(1, dtype=torch.int32, device=device)
    ms = timed(lambda: gdn.gdn_gate_projection(dims, hidden, w, a=a, b=b, d_status=status))
    ms_two = timed(lambda: (torch.matmul(hidden, w_a, out=a2), torch.matmul(hidden, w_b, out=b2)))
    # the two results agree to the bf16 rounding of the outputs
    torch.cuda.synchronize()
    agree = max(float((a.float() - a2.float()).abs().max()), float((b.float() - b2.float()).abs().max()))
    out_bytes = 2 * a.numel() * a.element_size()
    h_bytes = hidden.numel() * hidden.element_size()
    w_bytes = w.numel() * w.element_size()
    return {"ms": ms, "ms_two": ms_two, "bytes": h_bytes + w_bytes + out_bytes,
            "bytes_two": 2 * h_bytes + w_bytes + out_bytes, "d_model": inp["d_model"],
            "max_abs_diff_vs_library": agree, "status": int(status.item())}


def bench_slot_copy(torch, gdn, dims, device, steps, warmup, pairs=64):
    """Copy `pairs` whole slots (state and conv window) to `pairs` others in one
    call; the pool (2 x pairs slots, ~270 MB at the Qwen3.5-4B shape) is larger
    than L2."""
    io = torch.bfloat16 if dims.io == "bf16" else torch.float32
    n = 2 * pairs
    st = torch.randn((n, dims.h_v, dims.d_k, dims.d_v), device=device)
    cv = torch.randn((n, dims.conv_w - 1, gdn.conv_dim(dims)), device=device).to(io)
    src = torch.arange(pairs, dtype=torch.int32, device=device)
    dst = src + pairs
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for _ in range(max(warmup, 1)):
        gdn.gdn_slot_copy(dims, st, cv, src, dst, d_status=status)
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(steps)]
    for a_, b_ in ev:
        a_.record()
        gdn.gdn_slot_copy(dims, st, cv, src, dst, d_status=status)
        b_.record()
    torch.cuda.synchronize()
    ms = statistics.median(a_.elapsed_time(b_) for a_, b_ in ev)
    per_slot = st[0].numel() * 4 + cv[0].numel() * cv.element_size()
    return {"ms": ms, "bytes": 2 * pairs * per_slot, "pairs": pairs, "status": int(status.item())}


def bench_checkpointed(torch, gdn, run, steps, warmup, every=256):
    """The timed prefill again through gdn_prefill_checkpointed, leaving a
    checkpoint every `every` tokens (the interval PicoLM's server uses by
    default) in extra pool slots; L2 flushed before every timed step."""
    inp, d = run.inp, run.dims
    T = run.T
    n_ck = max(0, -(-T // every) - 1)
    base = run.state.shape[0]
    st = torch.cat([run.state, torch.zeros((n_ck,) + tuple(run.state.shape[1:]),
                                           device=run.state.device)])
    cv = torch.cat([run.conv, torch.zeros((n_ck,) + tuple(run.conv.shape[1:]), dtype=run.conv.dtype,
                                          device=run.conv.device)])
    ck = torch.tensor([base], dtype=torch.int32, device=run.state.device)
    flush = L2Flush(torch, run.state.device)

    def call():
        gdn.gdn_prefill_checkpointed(d, run.cw, run.A_log, run.dt_bias, run.x, run.a, run.b, run.cu,
                                     run.slot, run.init, st, cv, run.o, run.ws, every, ck,
                                     d_status=run.status)

    for _ in range(max(warmup, 1)):
        call()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk()) for _ in range(steps)]
    for a_, b_ in ev:
        flush()
        a_.record()
        call()
        b_.record()
    torch.cuda.synchronize()
    return {"ms": statistics.median(a_.elapsed_time(b_) for a_, b_ in ev), "every": every,
            "checkpoints": n_ck, "T": T, "status": int(run.status.item())}


def bench_fp32_state(torch, gdn, inp, device, steps, warmup):
    """The timed prefill with GDN_FP32_STATE (every product with the state in
    fp32: the SIMT path) on the same inputs; L2 flushed before every step."""
    import dataclasses
    run = Prefill(torch, gdn, dict(inp, dims=dataclasses.replace(inp["dims"], flags=gdn.GDN_FP32_STATE)),
                  device)
    flush = L2Flush(torch, device)
    for _ in range(max(warmup, 1)):
        run()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [{"s": mk(), "e": mk(), "b": [mk() for _ in gdn.STAGES], "f": [mk() for _ in gdn.STAGES]}
          for _ in range(steps)]
    stream = torch.cuda.current_stream()
    for e in ev:   # create the event handles before handing them to the library
        for x in [e["s"], e["e"], *e["b"], *e["f"]]:
            x.record(stream)
    torch.cuda.synchronize()
    for e in ev:
        flush()
        e["s"].record(stream)
        run()
        e["e"].record(stream)
    torch.cuda.synchronize()
    stage_ms, _ = trace_stages(torch, gdn, run, ev, flush)
    out = {"ms": statistics.median(e["s"].elapsed_time(e["e"]) for e in ev), "T": run.T,
           "stages_ms": stage_ms, "status": int(run.status.item())}
    del run
    return out


def bench_decode(torch, gdn, workloads, device, steps, warmup, layers=24, slots=64, graph=True):
    runs = []
    for layer in range(layers):
        inp = workloads.decode_4b(layer, slots=slots)
        d = inp["dims"]
        io = torch.bfloat16
        t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)  # noqa: E731
        runs.append(dict(dims=d, x=t(inp["x"], io), a=t(inp["a"], io), b=t(inp["b"], io),
                         cw=t(inp["conv_weight"]), A=t(inp["A_log"]), dt=t(inp["dt_bias"]),
                         slot=t(inp["slot_idx"]), state=t(inp["state_pool"]),
                         conv=t(inp["conv_pool"], io),
                         o=torch.empty((slots, d.h_v, d.d_v), dtype=io, device=device)))
    status = torch.zeros(1, dtype=torch.int32, device=device)

    def step():
        for r in runs:
            gdn.gdn_decode_step(r["dims"], r["cw"], r["A"], r["dt"], r["x"], r["a"], r["b"],
                                r["slot"], r["state"], r["conv"], r["o"], d_status=status)

    for _ in range(max(warmup, 1)):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [(mk(), mk()) for _ in range(steps)]
    # one timed per-layer call as well (the kernel's own launch duration)
    one = [(mk(), mk()) for _ in range(steps)]
    for (s, e), (s1, e1) in zip(evs, one):
        s.record(stream)
        for i, r in enumerate(runs):
            if i == 0:
                s1.record(stream)
            gdn.gdn_decode_step(r["dims"], r["cw"], r["A"], r["dt"], r["x"], r["a"], r["b"],
                                r["slot"], r["state"], r["conv"], r["o"], d_status=status)
            if i == 0:
                e1.record(stream)
        e.record(stream)
    torch.cuda.synchronize()
    step_ms = [s.elapsed_time(e) for s, e in evs]
    layer_ms = [s.elapsed_time(e) for s, e in one]
    # the same 24 calls captured once into a CUDA graph and replayed, as a
    # serving loop that captures its decode step launches them
    graph_ms, graph_err = (graph_replay_ms(torch, step, steps) if graph else
                           (None, "not captured with more than one rank"))
    d = runs[0]["dims"]
    state_bytes = 2 * layers * slots * d.h_v * d.d_k * d.d_v * 4
    norm = bench_decode_gated_norm(torch, gdn, runs, status, steps, warmup)
    return {"step_ms": step_ms, "layer_ms": layer_ms, "state_bytes": state_bytes,
            "layers": layers, "slots": slots, "status": int(status.item()), "gated_norm": norm,
            "graph_ms": graph_ms, "graph_err": graph_err}


def bench_decode_gated_norm(torch, gdn, runs, status, steps, warmup):
    """The same decode step with the gated RMSNorm of every layer's output:
    fused into the step (gdn_decode_step_gated_norm) and as the plain step plus
    the standalone norm per layer; median ms per 24-layer step of each."""
    d = runs[0]["dims"]
    dev = runs[0]["o"].device
    g = torch.Generator(device=dev).manual_seed(99)
    for r in runs:
        r["z"] = torch.randn(tuple(r["o"].shape), generator=g, device=dev).to(r["o"].dtype)
        r["w"] = torch.rand(d.d_v, generator=g, device=dev) + 0.5
        r["y"] = torch.empty_like(r["o"])

    def fused():
        for r in runs:
            gdn.gdn_decode_step_gated_norm(r["dims"], r["cw"], r["A"], r["dt"], r["x"], r["a"],
                                           r["b"], r["slot"], r["state"], r["conv"], r["z"],
                                           r["w"], r["y"], d_status=status)

    def unfused():
        for r in runs:
            gdn.gdn_decode_step(r["dims"], r["cw"], r["A"], r["dt"], r["x"], r["a"], r["b"],
                                r["slot"], r["state"], r["conv"], r["o"], d_status=status)
            gdn.gdn_gated_rmsnorm(r["dims"], r["w"], r["o"], r["z"], y=r["y"])

    out = {}
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for name, fn in (("fused", fused), ("unfused", unfused)):
        for _ in range(max(warmup, 1)):
            fn()
        evs = [(mk(), mk()) for _ in range(steps)]
        for a_, b_ in evs:
            a_.record()
            fn()
            b_.record()
        torch.cuda.synchronize()
        out[name + "_ms_per_step"] = statistics.median(a_.elapsed_time(b_) for a_, b_ in evs)
    out["saving_vs_unfused"] = 1.0 - out["fused_ms_per_step"] / out["unfused_ms_per_step"]
    return out


CPU_BASELINE_SECONDS = 10.0


def oracle_prefill_time(inp, n_threads):
    import oracle
    d = inp["dims"]
    ov = __import__("gated_deltanet_linear_07_gb300.workloads", fromlist=["x"]).oracle_view(inp)
    t0 = time.perf_counter()
    oracle.layer(inp["x"], inp["a"], inp["b"], inp["conv_weight"], inp["A_log"], inp["dt_bias"],
                 inp["cu_seqlens"], d.h_k, d.h_v, d.d_k, d.d_v, window0=ov["window0"],
                 state0=ov["state0"], l2_eps=d.l2_eps, n_threads=n_threads)
    return time.perf_counter() - t0


def prefill_dtype(d):
    """Arithmetic type of the prefill: the tensor-core path (Qwen3.5-4B layer
    shape, bf16 I/O) multiplies fp16 operands (bf16 with GDN_BF16_OPERANDS)
    with fp32 accumulation and an fp32 state; every other shape, and
    GDN_FP32_STATE, runs fp32 SIMT arithmetic."""
    tc = (d.d_k == 128 and d.d_v == 128 and d.chunk == 64 and d.io == "bf16" and
          d.h_v == 2 * d.h_k and not d.flags & 1)
    if not tc:
        return "f32"
    return "bf16" if d.flags & 8 else "fp16"


ARITHMETIC = {"fp16": "tensor-core products of fp16 operands (10-bit mantissa) with fp32 "
                      "accumulation; fp32 state, gates and norms; bf16 I/O",
              "bf16": "tensor-core products of bf16 operands with fp32 accumulation; fp32 "
                      "state, gates and norms; bf16 I/O",
              "f32": "fp32 SIMT arithmetic throughout"}


def config_of(inp):
    d = inp["dims"]
    return {"workload": "Qwen3.5-4B-shaped Gated DeltaNet layer prefill",
            "B": len(inp["lengths"]), "T": int(inp["x"].shape[0]), "h_k": d.h_k, "h_v": d.h_v,
            "d_k": d.d_k, "d_v": d.d_v, "conv_dim": d.conv_dim, "conv_w": d.conv_w,
            "chunk": d.chunk, "io": d.io, "state": "fp32, zero initial",
            "l2": "flushed before every timed step (256 MiB written, then 256 MiB read)",
            "timing": "median of the K timed steps (CUDA events per step)",
            "parallelism": "replicas (no cross-GPU exchange in the layer)"}


# ---------------------------------------------------------------- replicas

def max_over_ranks(dist, world, v, device):
    """The largest of each rank's value (one all-reduce; the value itself
    when there is one rank).  Timings take this so the slowest replica sets
    the job time."""
    if world == 1:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, units_per_rank, ms):
    """Whole-job units per second when every rank processes its own replica
    of `units_per_rank` units and the job takes `ms` milliseconds."""
    return world * units_per_rank / (ms / 1e3)


def prefill_roofline(d, T, stage, peak_tf, peak_src, reduce=lambda v: v, workload=None):
    """Roofline of the dominant prefill stage: the method's FLOPs that stage
    performs (per launch) over its event time, against the bf16 peak.  The
    chunk stage does K K^T, Q K^T, T (beta V), T (beta e^gamma K) (8 C d per
    token and head), the scan P W and Wk S^T, Q S^T, W^T K (2 C d + 6 d^2);
    in the overlapped launch the chunk work runs inside the scan stage's
    interval, which then carries both shares.  `workload` names a launch other
    than the T=4096 one, whose DRAM traffic is recorded under its own key."""
    stage_flops = {"frontend": 0.0,
                   "chunk": 8.0 * d.chunk * d.d_k * T * d.h_v,
                   "scan": (2.0 * d.chunk * d.d_k + 6.0 * d.d_k * d.d_k) * T * d.h_v}
    overlapped = "scan" in stage and "chunk" not in stage
    if overlapped:
        stage_flops["scan"] += stage_flops["chunk"]
    dom = max(stage, key=stage.get) if stage else None
    roof = None
    if dom and stage_flops.get(dom):
        dom_ms = reduce(stage[dom])
        ach = stage_flops[dom] / (dom_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": ach / peak_tf,
                "traffic": recorded_traffic(("prefill_overlap" if overlapped else "prefill_" + dom) +
                                            (":" + workload if workload else "")),
                "kernel": {"chunk": "prep_persistent_kernel (prefill stage 'chunk')",
                           "scan": ("scan_kernel (prefill stage 'scan')" if "chunk" in stage else
                                   "prep_persistent_kernel + scan_kernel, overlapped "
                                   "(prefill stage 'scan')")}.get(dom, dom),
                "peak_source": f"bf16_tflops ({peak_src})",
                "launch_ms": dom_ms, "flops_per_launch": stage_flops[dom]}
    stage_tflops = {k: stage_flops[k] / (v / 1e3) / 1e12 for k, v in stage.items()
                    if stage_flops.get(k)}
    return roof, stage_tflops


# ---------------------------------------------------------------- arms

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from gated_deltanet_linear_07_gb300 import workloads
    inp = workloads.prefill_4b()
    cores = os.cpu_count() or 1
    for _ in range(max(args.warmup, 0)):
        oracle_prefill_time(inp, cores)
    times = [oracle_prefill_time(inp, cores) for _ in range(args.steps)]
    T = inp["x"].shape[0]
    ms = 1e3 * statistics.median(times)   # the median, as the GPU arm takes
    value = T / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(inp),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"the whole workload ({T} tokens x 32 heads) per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gdn(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device visible"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    import gated_deltanet_linear_07_gb300 as gdn
    from gated_deltanet_linear_07_gb300 import workloads
    gdn.load()
    peaks, peak_src = load_peaks()
    sampler = ClockSampler(gpu_id_of(torch, local))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    sampler.start()
    time.sleep(0.2)
    pf = None
    if not args.no_prefill and not args.large_only:
        pf = bench_prefill(torch, gdn, workloads, device, args.steps, args.warmup)
        barrier()
    gn = gp = sc = ck = f32 = None
    if pf is not None:
        gn = bench_gated_norm(torch, gdn, pf["inp"]["dims"], pf["inp"]["x"].shape[0], device,
                              args.steps, args.warmup)
        barrier()
        gp = bench_gate_projection(torch, gdn, workloads, pf["inp"]["dims"],
                                   pf["inp"]["x"].shape[0], device, args.steps, args.warmup)
        barrier()
        sc = bench_slot_copy(torch, gdn, pf["inp"]["dims"], device, args.steps, args.warmup)
        barrier()
        ck = bench_checkpointed(torch, gdn, pf["run"], args.steps, args.warmup)
        barrier()
        f32 = bench_fp32_state(torch, gdn, pf["inp"], device, args.steps, args.warmup)
        barrier()
    large = {}
    if not args.no_large and not args.no_prefill:
        for name in LARGE_WORKLOADS:
            large[name] = bench_large(torch, gdn, workloads, device, name, args.steps, args.warmup,
                                      peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
                                      peak_src, peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
            barrier()
    dec = None
    if not args.no_decode and not args.large_only:
        dec = bench_decode(torch, gdn, workloads, device, args.decode_steps or args.steps,
                           args.warmup, layers=args.decode_layers, graph=world == 1)
        barrier()
    clocks = sampler.stop()
    if pf is None:
        if rank == 0 and large:
            print(json.dumps({"prefill_workloads": large, "clocks": clocks}), flush=True)
        if rank == 0 and dec is not None:
            print(json.dumps({"decode_only": True, "ms_per_step": statistics.median(dec["step_ms"]),
                              "layer_ms": statistics.median(dec["layer_ms"]),
                              "state_bytes": dec["state_bytes"], "clocks": clocks}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return 0
    e2e = None if args.no_e2e else bench_e2e(torch, gdn, pf["run"], args.steps, args.warmup)
    # CUDA-graph captures only in single-rank runs: a rank's process-group threads
    # keep working during a capture
    variants = None if args.no_variants or world > 1 else bench_launch_variants(
        torch, pf["run"], args.steps, device)

    def max_ranks(v):
        return max_over_ranks(dist, world, v, device)

    inp = pf["inp"]
    d = inp["dims"]
    T = inp["x"].shape[0]
    ms = max_ranks(statistics.median(pf["step_ms"]))   # median of the K steps
    value = replica_throughput(world, T, ms)
    flops_launch = alg_flops_per_token_head(d.chunk, d.d_k) * T * d.h_v
    peak_tf = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    roof, stage_tflops = prefill_roofline(d, T, pf["stage_ms"], peak_tf, peak_src, max_ranks)
    stage = pf["stage_ms"]
    if dec:   # collectives: every rank takes part
        dms = max_ranks(statistics.median(dec["step_ms"]))
        gms = max_ranks(dec["graph_ms"] if dec["graph_ms"] is not None else -1.0)
        lms = max_ranks(statistics.median(dec["layer_ms"]))
    out = None
    if rank == 0:
        hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": prefill_dtype(inp["dims"]), "arithmetic": ARITHMETIC[prefill_dtype(inp["dims"])],
            "data": "synthetic", "config": config_of(inp),
            "roofline": roof,
            "tc_roofline_frac_whole_step": flops_launch / (ms / 1e3) / 1e12 / peak_tf,
            "stages_ms": stage, "stages_tflops": stage_tflops,
            "gpu_launches": pf["launches"], "clocks": clocks,
            "device_status": pf["status"],
        }
        if large:
            line["prefill_workloads"] = large
        if variants:
            line["launch_variants"] = variants
        if e2e:
            line["e2e"] = {"value": replica_throughput(world, T, max_ranks(e2e["ms"])),
                           "unit": "tokens/s", "ms_per_step": e2e["ms"],
                           "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                           "pipeline": e2e["pipeline"], "link": e2e["link"],
                           "h2d_gbs_achieved": e2e["h2d"] / (e2e["ms"] / 1e3) / 1e9}
        if gn:
            ggbs = gn["bytes"] / (gn["ms"] / 1e3) / 1e9
            line["gated_norm"] = {
                "metric": "gated RMSNorm of the layer output, GB/s", "value": ggbs, "unit": "GB/s",
                "ms_per_call": gn["ms"],
                "config": {"workload": f"o, z [{T}, {d.h_v}, {d.d_v}] {d.io}, out of place",
                           "bytes_per_call": gn["bytes"],
                           "l2": "flushed before every timed call (256 MiB written, then 256 MiB read)"},
                "roofline": {"bound": "hbm", "achieved": ggbs, "peak": hbm, "unit": "GB/s",
                             "frac": ggbs / hbm, "traffic": recorded_traffic("gated_norm"),
                             "kernel": "gated_rmsnorm_kernel", "peak_source": f"hbm_gbs ({peak_src})",
                             "launch_ms": gn["ms"]}}
        if gp:
            pgbs = gp["bytes"] / (gp["ms"] / 1e3) / 1e9
            line["gate_projection"] = {
                "metric": "decay/beta input projections as one matmul, GB/s", "value": pgbs,
                "unit": "GB/s", "ms_per_call": gp["ms"],
                "config": {"workload": f"hidden [{T}, {gp['d_model']}] bf16 x [{2 * d.h_v}, "
                                       f"{gp['d_model']}] bf16 -> a, b [{T}, {d.h_v}] bf16",
                           "bytes_per_call": gp["bytes"],
                           "l2": "flushed before every timed call (256 MiB written, then 256 MiB read)"},
                "roofline": {"bound": "hbm", "achieved": pgbs, "peak": hbm, "unit": "GB/s",
                             "frac": pgbs / hbm, "traffic": recorded_traffic("gate_projection"),
                             "kernel": "gate_projection_kernel",
                             "peak_source": f"hbm_gbs ({peak_src})", "launch_ms": gp["ms"]},
                "vs_two_library_matmuls": {
                    "ms": gp["ms_two"], "launches": 2, "bytes": gp["bytes_two"],
                    "saved_launches": 1, "saved_bytes": gp["bytes_two"] - gp["bytes"],
                    "time_ratio": gp["ms_two"] / gp["ms"],
                    "max_abs_diff": gp["max_abs_diff_vs_library"]},
                "gpu_launches": 1, "device_status": gp["status"]}
        if sc:
            sgbs = sc["bytes"] / (sc["ms"] / 1e3) / 1e9
            line["slot_copy"] = {
                "metric": "slot copy (snapshot / restore) GB/s", "value": sgbs, "unit": "GB/s",
                "ms_per_call": sc["ms"],
                "config": {"workload": f"{sc['pairs']} slot pairs of the {T}-token layer's shape "
                                       f"(fp32 [{d.h_v}, {d.d_k}, {d.d_v}] state + conv window)",
                           "bytes_per_call": sc["bytes"],
                           "l2": "inputs larger than L2 (the pool is twice the copied bytes)"},
                "roofline": {"bound": "hbm", "achieved": sgbs, "peak": hbm, "unit": "GB/s",
                             "frac": sgbs / hbm, "traffic": recorded_traffic("slot_copy"),
                             "kernel": "slot_copy_kernel", "peak_source": f"hbm_gbs ({peak_src})",
                             "launch_ms": sc["ms"]},
                "device_status": sc["status"]}
        if ck:
            line["checkpointed_prefill"] = {
                "metric": "prefill tokens/s with interval checkpoints", "unit": "tokens/s",
                "value": ck["T"] / (ck["ms"] / 1e3), "ms_per_step": ck["ms"],
                "overhead_vs_plain": ck["ms"] / ms - 1.0,
                "config": {"workload": f"the timed prefill, a checkpoint every {ck['every']} tokens",
                           "checkpoints_per_step": ck["checkpoints"],
                           "l2": "flushed before every timed step"},
                "device_status": ck["status"]}
        if f32:
            line["fp32_state_prefill"] = {
                "metric": "prefill tokens/s with fp32 state products (GDN_FP32_STATE)",
                "unit": "tokens/s", "value": f32["T"] / (f32["ms"] / 1e3), "ms_per_step": f32["ms"],
                "slowdown_vs_tensor_core": f32["ms"] / ms, "stages_ms": f32["stages_ms"],
                "config": {"workload": "the timed prefill through the SIMT path, fp32 state products",
                           "l2": "flushed before every timed step"},
                "device_status": f32["status"]}
        if dec:
            # whole job: every rank moves its own replica's state bytes
            # the step as a serving loop runs it: its 24 calls replayed from one
            # CUDA graph (the plain back-to-back launches beside it)
            plain_gbs = replica_throughput(world, dec["state_bytes"], dms) / 1e9
            graphed = gms > 0
            step_ms = gms if graphed else dms
            gbs = replica_throughput(world, dec["state_bytes"], step_ms) / 1e9
            lgbs = dec["state_bytes"] / dec["layers"] / (lms / 1e3) / 1e9
            line["decode"] = {
                "metric": "decode state GB/s", "value": gbs, "unit": "GB/s",
                "ms_per_step": step_ms, "steps": args.decode_steps or args.steps,
                "launch": ("the 24 per-layer calls replayed from one CUDA graph" if graphed else
                           "the 24 per-layer calls launched back to back (no graph: "
                           f"{dec['graph_err']})"),
                "plain_launches": {"value": plain_gbs, "ms_per_step": dms},
                "config": {"workload": "decode step, 24 layers x 64 slots, one bf16 token per "
                                       "slot, shuffled slots, fp32 32x128x128 states",
                           "state_bytes_per_step": dec["state_bytes"],
                           "l2": "inputs larger than L2 (3.2 GB of state)"},
                "roofline": {"bound": "hbm", "achieved": lgbs, "peak": hbm, "unit": "GB/s",
                             "frac": lgbs / hbm, "traffic": recorded_traffic("decode_step"),
                             "kernel": "decode_step_kernel (one per-layer call)",
                             "peak_source": f"hbm_gbs ({peak_src})", "launch_ms": lms},
                "frac_whole_step": gbs / hbm, "gpu_launches": dec["layers"] * len(dec["step_ms"]),
                "gated_norm": dict(dec["gated_norm"], workload="the same step writing "
                                   "y = rmsnorm(o) * w * SiLU(z) for every layer"),
                "device_status": dec["status"]}
        if not args.no_cpu_baseline and world == 1:
            cores = os.cpu_count() or 1
            # whole-workload passes until about 10 s of oracle time have run
            passes, secs = 0, 0.0
            while passes == 0 or secs < CPU_BASELINE_SECONDS:
                secs += oracle_prefill_time(inp, cores)
                passes += 1
            line["cpu_baseline"] = {"value": passes * T / secs, "unit": "tokens/s",
                                    "cores": cores, "kind": "oracle",
                                    "sample": f"{passes} passes over the whole workload "
                                              f"({T} tokens x {d.h_v} heads each), {secs:.1f} s"}
        out = line
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gdn(args)


if __name__ == "__main__":
    sys.exit(main())
