"""C-ABI library: it builds for sm_103a, loads without a GPU, exports every
function include/gdn.h declares, and its host-side checks reject bad calls
before anything is launched (so these run on a CPU-only host: every call below
fails validation and never reaches the CUDA runtime)."""
import ctypes
import os
import re
import subprocess

import pytest

import gated_deltanet_linear_07_gb300 as gdn
from gated_deltanet_linear_07_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gdn.build()
    return gdn.load()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gdn_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_function(lib):
    declared = _declared()
    assert {"gdn_prefill", "gdn_decode_step", "gdn_conv1d_update",
            "gdn_prefill_workspace_size", "gdn_status_str"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln and "gdn_" in ln}
    assert exported == declared, exported ^ declared


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.gdn_status_str(code).decode() not in ("", "unknown status")
    assert lib.gdn_status_str(7).decode() == "unknown status"


D4B = dict(h_k=16, h_v=32, d_k=128, d_v=128, chunk=64, io="bf16")


def test_workspace_size_rules(lib):
    d = gdn.make_dims(**D4B)
    w1 = gdn.gdn_prefill_workspace_size(d, 4096, 1)
    w2 = gdn.gdn_prefill_workspace_size(d, 8192, 1)
    assert w1 > 0 and w2 > w1
    # tensor-core path (this shape): per chunk slot ([T/64] + B of them) one
    # 32 KiB [K;Q] tile per key head and a 41 KiB record per value head
    assert w1 >= (4096 // 64 + 1) * (16 * 32768 + 32 * 41984)
    # SIMT path (fp32 I/O): per token, fp32, the front end's normalised q, k, v and two
    # gates, and the chunk kernel's U, Wk, P rows and cumulative decay
    d32 = gdn.make_dims(**dict(D4B, io="fp32"))
    per_token = (2 * 16 * 128 + 32 * 128 + 2 * 32) + (32 * 128 + 32 * 128 + 32 * 64 + 32)
    assert gdn.gdn_prefill_workspace_size(d32, 4096, 1) >= 4096 * per_token * 4
    # chunk 128 on the SIMT path, at head dim 64 and at the 4B shape's 128 (streamed scan)
    for dd in (64, 128):
        assert gdn.gdn_prefill_workspace_size(gdn.make_dims(**dict(D4B, d_k=dd, d_v=dd, chunk=128)),
                                              4096, 1) > 0
    for bad in (dict(D4B, d_k=48), dict(D4B, chunk=256), dict(D4B, chunk=48), dict(D4B, h_v=33),
                dict(D4B, conv_w=3), dict(D4B, io=7), dict(D4B, h_k=1, h_v=65536, d_v=16)):
        assert gdn.gdn_prefill_workspace_size(gdn.make_dims(**bad), 4096, 1) == 0
    assert gdn.gdn_prefill_workspace_size(d, -1, 1) == 0
    # GDN_FP32_STATE moves this shape to the SIMT path: its per-token fp32 layout
    dfp = gdn.make_dims(**D4B, flags=gdn.GDN_FP32_STATE)
    assert gdn.gdn_prefill_workspace_size(dfp, 4096, 1) >= 4096 * (2 * 16 * 128 + 32 * 128 + 2 * 32) * 4
    assert gdn.gdn_prefill_workspace_size(dfp, 4096, 1) != w1
    # a call whose sequences are all empty takes the SIMT path (states and
    # windows pass through): no tensor-core chunk records
    w0 = gdn.gdn_prefill_workspace_size(d, 0, 3)
    assert 0 < w0 < 3 * (16 * 32768 + 32 * 41984)
    for bad_flags in (16, 32, -1):                 # unknown flag bits
        assert gdn.gdn_prefill_workspace_size(gdn.make_dims(**D4B, flags=bad_flags), 4096, 1) == 0
        assert _prefill(lib, gdn.make_dims(**D4B, flags=bad_flags)) == -1
    both = gdn.GDN_FP32_STATE | gdn.GDN_CHECK_FINITE
    assert gdn.gdn_prefill_workspace_size(gdn.make_dims(**D4B, flags=both), 4096, 1) == \
        gdn.gdn_prefill_workspace_size(dfp, 4096, 1)
    # the NaN/Inf probe reports through the device status word: none given
    assert _prefill(lib, gdn.make_dims(**D4B, flags=gdn.GDN_CHECK_FINITE)) == -1


FAKE = 1 << 20  # an aligned, never-dereferenced address: validation fails first


def _prefill(lib, dims, ws_bytes=1 << 40, ptrs=None, B=1, T=64, slots=1):
    p = _binding.gdn_params(FAKE, FAKE, FAKE)
    ptr = dict(x=FAKE, a=FAKE, b=FAKE, cu=FAKE, slot=FAKE, init=None, state=FAKE,
               conv=FAKE, o=FAKE, ws=FAKE)
    ptr.update(ptrs or {})
    return lib.gdn_prefill(ctypes.byref(dims), ctypes.byref(p), ptr["x"], ptr["a"], ptr["b"],
                           ptr["cu"], B, T, ptr["slot"], ptr["init"], ptr["state"], ptr["conv"],
                           slots, ptr["o"], ptr["ws"], ws_bytes, None, None)


def test_prefill_rejects_bad_calls_before_launch(lib):
    d = gdn.make_dims(**D4B)
    assert _prefill(lib, gdn.make_dims(**dict(D4B, d_k=48))) == -2
    assert _prefill(lib, gdn.make_dims(**dict(D4B, h_v=24))) == -1
    assert _prefill(lib, d, ptrs=dict(cu=None)) == -1
    assert _prefill(lib, d, ptrs=dict(state=None)) == -1
    assert _prefill(lib, d, ptrs=dict(x=None)) == -1
    assert _prefill(lib, d, ws_bytes=16) == -4
    assert _prefill(lib, d, ptrs=dict(ws=None)) == -4
    assert _prefill(lib, d, ptrs=dict(x=FAKE + 2)) == -5
    assert _prefill(lib, d, ptrs=dict(state=FAKE + 4)) == -5
    assert _prefill(lib, d, ptrs=dict(ws=FAKE + 16)) == -5
    assert _prefill(lib, d, B=-1) == -1
    assert _prefill(lib, d, B=0, T=5) == -1
    assert _prefill(lib, d, B=0, T=0) == 0        # empty batch: nothing to do


def test_decode_and_conv_reject_bad_calls_before_launch(lib):
    d = gdn.make_dims(**D4B)
    p = _binding.gdn_params(FAKE, FAKE, FAKE)
    call = lambda **kw: lib.gdn_decode_step(  # noqa: E731
        ctypes.byref(kw.get("dims", d)), ctypes.byref(p), kw.get("x", FAKE), FAKE, FAKE, FAKE,
        kw.get("n", 4), kw.get("state", FAKE), FAKE, 8, kw.get("o", FAKE), None, None)
    assert call(dims=gdn.make_dims(**dict(D4B, d_v=24))) == -2
    assert call(x=None) == -1
    assert call(n=-1) == -1
    assert call(n=0) == 0
    assert call(o=FAKE + 8) == -5
    assert call(state=FAKE + 12) == -5
    assert lib.gdn_conv1d_update(ctypes.byref(d), FAKE, None, FAKE, 8, FAKE, 4, FAKE, None,
                                 None) == -1
    assert lib.gdn_conv1d_update(ctypes.byref(d), FAKE + 4, FAKE, FAKE, 8, FAKE, 4, FAKE, None,
                                 None) == -5
    assert lib.gdn_conv1d_update(ctypes.byref(d), FAKE, FAKE, FAKE, 8, FAKE, 0, FAKE, None,
                                 None) == 0


def test_gated_rmsnorm_rejects_bad_calls_before_launch(lib):
    d = gdn.make_dims(**D4B)
    call = lambda **kw: lib.gdn_gated_rmsnorm(  # noqa: E731
        ctypes.byref(kw.get("dims", d)), kw.get("w", FAKE), ctypes.c_float(kw.get("eps", 1e-6)),
        kw.get("o", FAKE), kw.get("z", FAKE), kw.get("n", 4), kw.get("y", FAKE), None)
    assert call(dims=gdn.make_dims(**dict(D4B, d_v=48))) == -2
    assert call(o=None) == -1
    assert call(z=None) == -1
    assert call(n=-1) == -1
    assert call(eps=-1.0) == -1
    assert call(eps=float("nan")) == -1
    assert call(n=0) == 0
    assert call(w=FAKE + 4) == -5
    assert call(y=FAKE + 8) == -5


def test_gate_projection_rejects_bad_calls_before_launch(lib):
    d = gdn.make_dims(**D4B)
    call = lambda **kw: lib.gdn_gate_projection(  # noqa: E731
        ctypes.byref(kw.get("dims", d)) if kw.get("dims", d) is not None else None,
        kw.get("hidden", FAKE), kw.get("w", FAKE), kw.get("d_model", 2560), kw.get("n", 4),
        kw.get("a", FAKE), kw.get("b", FAKE), None, None)
    assert call(dims=None) == -1
    assert call(n=-1) == -1
    assert call(d_model=0) == -1
    assert call(hidden=None) == -1
    assert call(b=None) == -1
    assert call(dims=gdn.make_dims(**dict(D4B, h_k=1, h_v=8))) == -2    # h_v not a multiple of 16
    assert call(dims=gdn.make_dims(**dict(D4B, h_k=16, h_v=144))) == -2  # 2 h_v above 256
    assert call(d_model=2500) == -2                                      # not a multiple of 64
    assert call(n=1 << 31) == -2                                         # above 2^31 - 1 tokens
    assert call(n=0) == 0
    assert call(hidden=FAKE + 2) == -5
    assert call(a=FAKE + 8) == -5


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _binding.load()


def test_slot_copy_and_checkpointed_prefill_reject_bad_calls_before_launch(lib):
    d = gdn.make_dims(**D4B)
    copy = lambda **kw: lib.gdn_slot_copy(  # noqa: E731
        ctypes.byref(kw.get("dims", d)), kw.get("state", FAKE), kw.get("conv", FAKE), 8,
        kw.get("src", FAKE), kw.get("dst", FAKE), kw.get("n", 4), None, None)
    assert copy(dims=gdn.make_dims(**dict(D4B, d_v=48))) == -2
    assert copy(src=None) == -1
    assert copy(dst=None) == -1
    assert copy(state=None) == -1
    assert copy(n=-1) == -1
    assert copy(n=0) == 0                          # nothing to copy
    assert copy(state=FAKE + 4) == -5
    assert copy(conv=FAKE + 8) == -5
    p = _binding.gdn_params(FAKE, FAKE, FAKE)

    def ck(dims=d, every=128, ckpt=FAKE, cu=FAKE, x=FAKE):
        return lib.gdn_prefill_checkpointed(
            ctypes.byref(dims), ctypes.byref(p), x, FAKE, FAKE, cu, 1, 64, FAKE, None, FAKE,
            FAKE, 1, FAKE, FAKE, 1 << 40, every, ckpt, None, None)
    assert ck(dims=gdn.make_dims(**dict(D4B, d_k=48))) == -2
    assert ck(every=0) == -1
    assert ck(every=-64) == -1
    assert ck(every=96) == -1                      # not a multiple of the chunk (64)
    assert ck(ckpt=None) == -1
    assert ck(cu=None) == -1                       # and every gdn_prefill check still applies
    assert ck(x=FAKE + 2) == -5


def test_fused_gated_norm_variants_reject_bad_calls_before_launch(lib):
    d = gdn.make_dims(**D4B)
    p = _binding.gdn_params(FAKE, FAKE, FAKE)
    Z, Y = FAKE + 4096, FAKE + 8192

    def pf(dims=d, z=Z, w=FAKE, eps=1e-6, y=Y, T=64, cu=FAKE):
        return lib.gdn_prefill_gated_norm(
            ctypes.byref(dims), ctypes.byref(p), FAKE, FAKE, FAKE, cu, 1, T, FAKE, None, FAKE,
            FAKE, 1, z, w, ctypes.c_float(eps), y, FAKE, 1 << 40, None, None)
    assert pf(dims=gdn.make_dims(**dict(D4B, d_v=48))) == -2
    assert pf(z=None) == -1
    assert pf(w=None) == -1
    assert pf(eps=-1.0) == -1
    assert pf(eps=float("nan")) == -1
    assert pf(y=Z) == -1                           # y may not alias z
    assert pf(z=Z + 8) == -5
    assert pf(w=FAKE + 4) == -5
    assert pf(y=Y + 2) == -5                       # y is the layer's output buffer
    assert pf(cu=None) == -1                       # and every gdn_prefill check still applies

    def dc(z=Z, w=FAKE, eps=1e-6, y=Y, n=4):
        return lib.gdn_decode_step_gated_norm(
            ctypes.byref(d), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, n, FAKE, FAKE, 8, z, w,
            ctypes.c_float(eps), y, None, None)
    assert dc(z=None) == -1
    assert dc(w=None) == -1
    assert dc(eps=float("nan")) == -1
    assert dc(y=Z) == -1
    assert dc(z=Z + 8) == -5
    assert dc(y=Y + 4) == -5
    assert dc(n=0) == 0                            # nothing to do
