"""Seeded synthetic inputs for the Gated DeltaNet layer.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic.  Both the CUDA path's tests/benchmark and the float64
oracle read the arrays it returns, so the two sides always see identical
inputs.  Values meant for a bf16 boundary are rounded to bf16 here (round to
nearest even) and kept as float32, so widening them for the oracle is exact and
converting them to torch.bfloat16 for the GPU is exact too.

Workloads (numpy PCG64, workload i uses seed 1000 + i):
  1 tiny         1 seq, T=64, H_k=H_v=2, d_k=d_v=16, fp32, chunk 16, zero state.
  2 prefill_4b   1 seq, T=4096, Qwen3.5-4B layer shape (H_k=16, H_v=32,
                 d=128, conv over 8192 channels), bf16, chunk 64, zero state.
  3 decode_4b    24 layers x 64 slots, states ~ N(0, 0.02^2) fp32, windows
                 ~ N(0,1) bf16, one bf16 token per slot, shuffled slots.
  4 adversarial  4 seqs x T=32768, 4B shape, bf16, random initial state and
                 window; key channels alternate 512-token runs of one repeated
                 vector with 512-token random segments; b ~ N(6,1) so beta is
                 near 1.  Sub-case "b" also pins a = -12 (decay near 1).
  5 varlen       16 seqs, lengths ~ U{1..8192}, 4B shape, bf16, shuffled slots,
                 then 256 decode tokens per sequence.
  6 gate_projection_inputs  hidden states [n][2560] ~ N(0,1) and the decay/beta
                 projection weights [2 H_v][2560] ~ N(0, 1/2560), both bf16, so
                 that the projected a and b are ~ N(0,1) like the layer's.
Distributions: x, a, b ~ N(0,1) unless stated; conv weight ~ N(0, 0.5^2);
A_log ~ U(0, 2.7); dt_bias ~ N(0, 0.1^2).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 1000


@dataclass(frozen=True)
class Dims:
    h_k: int
    h_v: int
    d_k: int
    d_v: int
    conv_w: int = 4
    chunk: int = 64
    io: str = "bf16"          # "fp32" | "bf16"
    l2_eps: float = 1e-6
    flags: int = 0            # gdn_dims.flags (GDN_FP32_STATE)

    @property
    def conv_dim(self) -> int:
        return 2 * self.h_k * self.d_k + self.h_v * self.d_v


TINY = Dims(h_k=2, h_v=2, d_k=16, d_v=16, chunk=16, io="fp32")
QWEN35_4B = Dims(h_k=16, h_v=32, d_k=128, d_v=128, chunk=64, io="bf16")


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), kept as float32.
    Works in place on a float32 copy, in slices, with 32-bit integer arithmetic
    (finite inputs only)."""
    out = np.array(a, dtype=np.float32, copy=True, order="C")
    flat = out.reshape(-1).view(np.uint32)
    step = 1 << 24
    for i in range(0, flat.size, step):
        u = flat[i:i + step]
        u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
        u &= np.uint32(0xFFFF0000)
    return out


def _io(a: np.ndarray, dims: Dims) -> np.ndarray:
    return round_bf16(a) if dims.io == "bf16" else np.ascontiguousarray(a, np.float32)


def _normal(rng, shape, std=1.0, mean=0.0):
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    if mean != 0.0:
        out += np.float32(mean)
    return out


def params(rng, dims: Dims) -> dict:
    """Layer parameters: conv weight [conv_dim][W], A_log, dt_bias [h_v] (fp32)."""
    return {
        "conv_weight": _normal(rng, (dims.conv_dim, dims.conv_w), std=0.5),
        "A_log": rng.uniform(0.0, 2.7, size=dims.h_v).astype(np.float32),
        "dt_bias": _normal(rng, (dims.h_v,), std=0.1),
    }


def layer_inputs(dims: Dims, lengths, seed: int, *, init: str = "zero",
                 num_slots: int | None = None, shuffle_slots: bool = True,
                 b_mean: float = 0.0, a_const: float | None = None,
                 state_std: float = 0.02, correlated_keys: int = 0) -> dict:
    """Inputs of one varlen prefill call.

    init: "zero" (no initial state; the slots hold junk that must be ignored),
    "random" (every sequence starts from a random state and window), or
    "mixed" (alternating).  correlated_keys=R > 0 makes the key channels of x
    alternate R-token runs of one repeated vector with R-token random segments.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = [int(t) for t in lengths]
    B = len(lengths)
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    T_tot = int(cu[-1])
    if num_slots is None:
        num_slots = max(B, 1) + 3
    p = params(rng, dims)
    x = _normal(rng, (T_tot, dims.conv_dim))
    if correlated_keys:
        R = int(correlated_keys)
        k0, k1 = dims.h_k * dims.d_k, 2 * dims.h_k * dims.d_k
        for s in range(B):
            start, T = int(cu[s]), lengths[s]
            for r0 in range(0, T, 2 * R):
                r1 = min(r0 + R, T)
                vec = _normal(rng, (k1 - k0,))
                x[start + r0:start + r1, k0:k1] = vec[None, :]
    a = _normal(rng, (T_tot, dims.h_v))
    if a_const is not None:
        a[:] = np.float32(a_const)
    b = _normal(rng, (T_tot, dims.h_v), mean=b_mean)
    perm = rng.permutation(num_slots) if shuffle_slots else np.arange(num_slots)
    slot_idx = perm[:B].astype(np.int32)
    if init == "zero":
        has_init = np.zeros(B, np.uint8)
    elif init == "random":
        has_init = np.ones(B, np.uint8)
    elif init == "mixed":
        has_init = (np.arange(B) % 2 == 0).astype(np.uint8)
    else:
        raise ValueError(init)
    # Pool contents: random everywhere (sequences without an initial state must
    # ignore what their slot holds).
    state_pool = _normal(rng, (num_slots, dims.h_v, dims.d_k, dims.d_v), std=state_std)
    conv_pool = _io(_normal(rng, (num_slots, dims.conv_w - 1, dims.conv_dim)), dims)
    return {
        "dims": dims, "x": _io(x, dims), "a": _io(a, dims), "b": _io(b, dims),
        "cu_seqlens": cu, "lengths": lengths, "slot_idx": slot_idx,
        "has_init": has_init, "num_slots": num_slots,
        "state_pool": state_pool, "conv_pool": conv_pool, **p,
    }


def oracle_view(inp: dict) -> dict:
    """Per-sequence initial state / window (zeros where a sequence has no
    initial state), gathered from the slot pools: the arrays the oracle takes."""
    dims: Dims = inp["dims"]
    B = len(inp["lengths"])
    st = np.zeros((B, dims.h_v, dims.d_k, dims.d_v), np.float32)
    win = np.zeros((B, dims.conv_w - 1, dims.conv_dim), np.float32)
    for s in range(B):
        if inp["has_init"][s]:
            st[s] = inp["state_pool"][inp["slot_idx"][s]]
            win[s] = inp["conv_pool"][inp["slot_idx"][s]]
    return {"state0": st, "window0": win}


def decode_inputs(dims: Dims, n_rows: int, num_slots: int, seed: int,
                  state_std: float = 0.02, padding_rows: int = 0) -> dict:
    """One decode step: n_rows tokens, each for a distinct slot (shuffled).
    padding_rows of them (at random positions) carry slot -1."""
    rng = np.random.Generator(np.random.PCG64(seed))
    p = params(rng, dims)
    x = _io(_normal(rng, (n_rows, dims.conv_dim)), dims)
    a = _io(_normal(rng, (n_rows, dims.h_v)), dims)
    b = _io(_normal(rng, (n_rows, dims.h_v)), dims)
    slot_idx = rng.permutation(num_slots)[:n_rows].astype(np.int32)
    if padding_rows:
        pad = rng.choice(n_rows, size=padding_rows, replace=False)
        slot_idx[pad] = -1
    state_pool = _normal(rng, (num_slots, dims.h_v, dims.d_k, dims.d_v), std=state_std)
    conv_pool = _io(_normal(rng, (num_slots, dims.conv_w - 1, dims.conv_dim)), dims)
    return {"dims": dims, "x": x, "a": a, "b": b, "slot_idx": slot_idx,
            "num_slots": num_slots, "state_pool": state_pool,
            "conv_pool": conv_pool, **p}


# ---- the five named workloads -------------------------------------------

def tiny(seed: int = SEED_BASE + 1) -> dict:
    return layer_inputs(TINY, [64], seed, init="zero", num_slots=1,
                        shuffle_slots=False)


def prefill_4b(seed: int = SEED_BASE + 2, T: int = 4096) -> dict:
    return layer_inputs(QWEN35_4B, [T], seed, init="zero", num_slots=1,
                        shuffle_slots=False)


def decode_4b(layer: int, seed: int = SEED_BASE + 3, slots: int = 64) -> dict:
    """Layer `layer` (0..23) of the 24-layer decode step."""
    return decode_inputs(QWEN35_4B, slots, slots, seed * 100 + layer)


def adversarial(seed: int = SEED_BASE + 4, B: int = 4, T: int = 32768,
                sub: str = "a") -> dict:
    return layer_inputs(QWEN35_4B, [T] * B, seed + (100 if sub == "b" else 0),
                        init="random", num_slots=B, b_mean=6.0,
                        a_const=(-12.0 if sub == "b" else None),
                        correlated_keys=512)


def varlen_lengths(seed: int = SEED_BASE + 5, B: int = 16, max_len: int = 8192):
    """The sequence lengths of the mixed varlen batch, U{1..max_len}, and the
    generator that drew them (its later draws are the decode tokens)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(1, max_len + 1, size=B), rng


def varlen(seed: int = SEED_BASE + 5, B: int = 16, max_len: int = 8192,
           decode_steps: int = 256) -> dict:
    lengths, rng = varlen_lengths(seed, B, max_len)
    inp = layer_inputs(QWEN35_4B, lengths, seed + 1, init="zero", num_slots=B)
    dims = inp["dims"]
    inp["decode_x"] = _io(_normal(rng, (decode_steps, B, dims.conv_dim)), dims)
    inp["decode_a"] = _io(_normal(rng, (decode_steps, B, dims.h_v)), dims)
    inp["decode_b"] = _io(_normal(rng, (decode_steps, B, dims.h_v)), dims)
    return inp


# The model width the decay/beta projection reads at the 4B shape (the
# Qwen3-4B family's hidden size).
D_MODEL_4B = 2560


def gate_projection_inputs(n: int, d_model: int = D_MODEL_4B, h_v: int = 32,
                           seed: int = SEED_BASE + 6) -> dict:
    """Inputs of the decay/beta projection: hidden [n][d_model] ~ N(0,1) and
    w_ba [2 h_v][d_model] ~ N(0, 1/d_model) (decay rows, then beta rows), both
    rounded to bf16 and kept as float32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return {"hidden": round_bf16(_normal(rng, (n, d_model))),
            "w_ba": round_bf16(_normal(rng, (2 * h_v, d_model), std=float(d_model) ** -0.5)),
            "h_v": h_v, "d_model": d_model}
