"""Pins of the float64 oracle against things other than itself.

Each test ties one part of the oracle to an independent fact: the unrolled
closed form on tiny inputs (brute force), an independent chunked evaluation,
closed forms (pure decay, exact key-to-value recall, repeated-key overwrite,
the identical-key chunk inverse), library routines (np.convolve, expit,
logaddexp, norms) for the front end, and invariants (handoff, varlen leak,
contraction bound).  A plausible slip in the oracle -- a transposed state, a
dropped decay, an off-by-one in the conv window, the wrong key head -- breaks at
least one of them.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from tests._independent import brute_force, chunk_inverse, chunked_wy

RNG = np.random.default_rng


def _unit_rows(a):
    return a / np.linalg.norm(a, axis=1, keepdims=True)


def _rand_head(rng, T, d_k, d_v, g_scale=0.3):
    k = _unit_rows(rng.standard_normal((T, d_k)))
    q = _unit_rows(rng.standard_normal((T, d_k))) / np.sqrt(d_k)
    v = rng.standard_normal((T, d_v))
    g = -g_scale * rng.random(T)
    beta = rng.random(T)
    S0 = rng.standard_normal((d_v, d_k))  # deliberately non-symmetric / non-square
    return q, k, v, g, beta, S0


# ---------------------------------------------------------------- recurrence

@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("d_k,d_v", [(4, 4), (3, 5), (6, 2)])
def test_recurrence_matches_brute_force(T, d_k, d_v):
    q, k, v, g, beta, S0 = _rand_head(RNG(T * 100 + d_k * 10 + d_v), T, d_k, d_v)
    o_ref, S_ref = brute_force(q, k, v, g, beta, S0)
    o, S = oracle.recurrence(q, k, v, g, beta, S0)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * max(1, np.abs(o_ref).max()))
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12 * max(1, np.abs(S_ref).max()))


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_recurrence_matches_independent_chunked_form(C):
    q, k, v, g, beta, S0 = _rand_head(RNG(7 + C), 37, 8, 12)
    o_ref, S_ref = chunked_wy(q, k, v, g, beta, S0, C=C)
    o, S = oracle.recurrence(q, k, v, g, beta, S0)
    assert np.abs(o - o_ref).max() <= 1e-10 * np.abs(o_ref).max()
    assert np.abs(S - S_ref).max() <= 1e-10 * np.abs(S_ref).max()


@pytest.mark.parametrize("C", [32, 64, 128])
def test_recurrence_matches_chunked_form_at_the_gpu_chunk_lengths(C):
    """The same independent chunked evaluation at the chunk lengths the GPU
    paths run (several full chunks and a ragged tail): the chunk length only
    changes rounding."""
    q, k, v, g, beta, S0 = _rand_head(RNG(70 + C), 300, 8, 12)
    o_ref, S_ref = chunked_wy(q, k, v, g, beta, S0, C=C)
    o, S = oracle.recurrence(q, k, v, g, beta, S0)
    assert np.abs(o - o_ref).max() <= 1e-10 * np.abs(o_ref).max()
    assert np.abs(S - S_ref).max() <= 1e-10 * np.abs(S_ref).max()


def test_beta_zero_is_pure_decay():
    """beta = 0: S_T = exp(sum g) S_0 and o_t = exp(sum_{s<=t} g_s) S_0 q_t."""
    q, k, v, g, _, S0 = _rand_head(RNG(11), 20, 8, 6, g_scale=2.0)
    beta = np.zeros(20)
    o, S = oracle.recurrence(q, k, v, g, beta, S0)
    cum = np.cumsum(g)
    np.testing.assert_allclose(S, np.exp(cum[-1]) * S0, rtol=1e-13, atol=0)
    np.testing.assert_allclose(o, np.exp(cum)[:, None] * (q @ S0.T), rtol=1e-12, atol=1e-300)


def test_orthonormal_keys_give_exact_recall():
    """alpha = 1, beta = 1, orthonormal keys from S_0 = 0: S k_j = v_j, so a
    query equal to k_j reads back v_j exactly."""
    d = 12
    rng = RNG(5)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    keys = Qm.T                        # rows orthonormal
    vals = rng.standard_normal((d, 7))
    g = np.zeros(d)
    beta = np.ones(d)
    # the query of token t asks for the key written one token earlier
    queries = np.roll(keys, 1, axis=0)
    o, S = oracle.recurrence(queries, keys, vals, g, beta, None)
    np.testing.assert_allclose(S @ keys.T, vals.T, atol=1e-12)
    np.testing.assert_allclose(o[1:], vals[:-1], atol=1e-12)


def test_repeated_key_with_beta_one_overwrites():
    """beta = 1 and the same key every token: S_t k = v_t for any S_{t-1}, decay."""
    rng = RNG(9)
    d_k, d_v, T = 10, 6, 15
    kvec = _unit_rows(rng.standard_normal((1, d_k)))[0]
    k = np.tile(kvec, (T, 1))
    v = rng.standard_normal((T, d_v))
    g = -rng.random(T)
    o, S = oracle.recurrence(k, k, v, g, np.ones(T), rng.standard_normal((d_v, d_k)))
    np.testing.assert_allclose(o, v, atol=1e-12)
    np.testing.assert_allclose(S @ kvec, v[-1], atol=1e-12)


def test_identical_key_chunk_inverse_closed_form():
    """Identical unit keys, beta_s = b: (I + A)^-1 has 1 on the diagonal and
    -b (1-b)^{s-j-1} exp(gamma_s - gamma_j) below it.  Pins the chunked
    evaluator used above on the fully correlated case the oxydllm notes (New
    Features, "Gated DeltaNet runtime") report as the overflow trap."""
    C = 64
    rng = RNG(3)
    for b in (1.0, 0.9975, 0.3):
        k = np.tile(_unit_rows(rng.standard_normal((1, 32))), (C, 1))
        g = -0.05 * rng.random(C)
        Tm = chunk_inverse(k, g, np.full(C, b))
        gam = np.cumsum(g)
        s, j = np.meshgrid(np.arange(C), np.arange(C), indexing="ij")
        expect = np.where(s == j, 1.0, np.where(
            j < s, -b * (1 - b) ** np.maximum(s - j - 1, 0) * np.exp(gam[s] - gam[j]), 0.0))
        np.testing.assert_allclose(Tm, expect, atol=1e-9)
        assert np.abs(Tm).max() <= 1.0 + 1e-9


def test_state_norm_contraction_bound():
    """||S_t||_2 <= alpha_t ||S_{t-1}||_2 + beta_t ||v_t||: I - beta k k^T is a
    contraction for beta in [0, 2] and unit k."""
    q, k, v, g, beta, S = _rand_head(RNG(21), 30, 8, 8)
    for t in range(30):
        _, S_new = oracle.recurrence(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                     beta[t:t + 1], S)
        bound = np.exp(g[t]) * np.linalg.norm(S, 2) + beta[t] * np.linalg.norm(v[t])
        assert np.linalg.norm(S_new, 2) <= bound * (1 + 1e-12)
        S = S_new


# ------------------------------------------------------------------ front end

def _layer_case(seed, h_k=2, h_v=4, d_k=8, d_v=6, lengths=(13,), with_init=True):
    rng = RNG(seed)
    cd = 2 * h_k * d_k + h_v * d_v
    T = int(sum(lengths))
    B = len(lengths)
    return dict(
        x=rng.standard_normal((T, cd)).astype(np.float32),
        a=rng.standard_normal((T, h_v)).astype(np.float32),
        b=rng.standard_normal((T, h_v)).astype(np.float32),
        conv_weight=(0.5 * rng.standard_normal((cd, 4))).astype(np.float32),
        A_log=rng.uniform(0, 2.7, h_v).astype(np.float32),
        dt_bias=(0.1 * rng.standard_normal(h_v)).astype(np.float32),
        cu_seqlens=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
        window0=(rng.standard_normal((B, 3, cd)).astype(np.float32) if with_init else None),
        state0=((0.1 * rng.standard_normal((B, h_v, d_k, d_v))).astype(np.float32)
                if with_init else None),
        h_k=h_k, h_v=h_v, d_k=d_k, d_v=d_v)


def test_conv_silu_matches_numpy_convolve_and_expit():
    c = _layer_case(1)
    x, w, win = c["x"], c["conv_weight"], c["window0"][0]
    y = oracle.conv_silu(x, w, win)
    xt = np.concatenate([win, x]).astype(np.float64)
    for ch in range(x.shape[1]):
        z = np.convolve(xt[:, ch], w[ch, ::-1].astype(np.float64), mode="valid")
        np.testing.assert_allclose(y[:, ch], z * expit(z), rtol=1e-13, atol=1e-15)
    # without a window the history is zero
    y0 = oracle.conv_silu(x, w, None)
    xt0 = np.concatenate([np.zeros_like(win), x]).astype(np.float64)
    z = np.convolve(xt0[:, 5], w[5, ::-1].astype(np.float64), mode="valid")
    np.testing.assert_allclose(y0[:, 5], z * expit(z), rtol=1e-13, atol=1e-15)


def test_conv_impulse_response_is_the_taps_in_reverse_time():
    cd = 2 * 1 * 4 + 1 * 4
    w = RNG(2).standard_normal((cd, 4)).astype(np.float32)
    x = np.zeros((10, cd), np.float32)
    x[3, :] = 1.0
    y = oracle.conv_silu(x, w, None)
    z = np.zeros((10, cd))
    for lag in range(4):       # token 3 + lag sees the impulse through tap 3 - lag
        z[3 + lag] = w[:, 3 - lag]
    np.testing.assert_allclose(y, z * expit(z), rtol=1e-13, atol=1e-15)


def test_frontend_gates_norms_and_head_split():
    c = _layer_case(4)
    h_k, h_v, d_k, d_v = c["h_k"], c["h_v"], c["d_k"], c["d_v"]
    y = oracle.conv_silu(c["x"], c["conv_weight"], c["window0"][0])
    for h in range(h_v):
        qh, kh, vv, g, be = oracle.frontend_head(
            c["x"], c["a"], c["b"], c["conv_weight"], c["A_log"], c["dt_bias"],
            h_k, h_v, d_k, d_v, h, window0=c["window0"][0])
        hk = h // (h_v // h_k)
        yq = y[:, hk * d_k:(hk + 1) * d_k]
        yk = y[:, h_k * d_k + hk * d_k:h_k * d_k + (hk + 1) * d_k]
        yv = y[:, 2 * h_k * d_k + h * d_v:2 * h_k * d_k + (h + 1) * d_v]
        np.testing.assert_allclose(vv, yv, rtol=1e-15, atol=0)
        # unit keys (up to eps), queries of norm 1/sqrt(d_k), same directions
        nk = np.linalg.norm(yk, axis=1)
        np.testing.assert_allclose(np.linalg.norm(kh, axis=1), nk / np.sqrt(nk ** 2 + 1e-6), rtol=1e-14)
        np.testing.assert_allclose(kh * nk[:, None] / np.linalg.norm(kh, axis=1)[:, None], yk, rtol=1e-12, atol=1e-14)
        nq = np.linalg.norm(yq, axis=1)
        np.testing.assert_allclose(np.linalg.norm(qh, axis=1) * np.sqrt(d_k), nq / np.sqrt(nq ** 2 + 1e-6), rtol=1e-14)
        np.testing.assert_allclose(qh * nq[:, None] / np.linalg.norm(qh, axis=1)[:, None], yq, rtol=1e-12, atol=1e-14)
        # gates: g = -exp(A_log) softplus(a + dt_bias) <= 0; beta = sigmoid(b)
        z = c["a"][:, h].astype(np.float64) + np.float64(c["dt_bias"][h])
        np.testing.assert_allclose(g, -np.exp(np.float64(c["A_log"][h])) * np.logaddexp(0.0, z), rtol=1e-14)
        np.testing.assert_allclose(be, expit(c["b"][:, h].astype(np.float64)), rtol=1e-15)
        assert (g <= 0).all() and ((be > 0) & (be < 1)).all()


def _recall_layer(h_k, h_v, d):
    """Inputs whose front end yields standard-basis keys and queries: conv taps
    (0,0,0,1), x = 10 e_m on the key/query channels, a = -100 (decay 1),
    b = 40 (beta 1).  Key head hk writes key e_{perm_hk[t]} at token t and the
    query of token t asks for the key of token t-1."""
    rng = RNG(17)
    T = d
    cd = 2 * h_k * d + h_v * d
    x = np.zeros((T, cd), np.float32)
    perms = [rng.permutation(d) for _ in range(h_k)]
    for hk in range(h_k):
        for t in range(T):
            x[t, h_k * d + hk * d + perms[hk][t]] = 10.0
            if t > 0:
                x[t, hk * d + perms[hk][t - 1]] = 10.0
    x[:, 2 * h_k * d:] = rng.standard_normal((T, h_v * d)).astype(np.float32)
    w = np.zeros((cd, 4), np.float32)
    w[:, 3] = 1.0
    a = np.full((T, h_v), -100.0, np.float32)
    b = np.full((T, h_v), 40.0, np.float32)
    return x, a, b, w


def test_layer_recall_through_the_front_end_and_key_head_mapping():
    """Exact recall through the whole layer, and value head h reading key head
    h // (H_v/H_k): heads of one key group recall that group's keys only."""
    h_k, h_v, d = 2, 4, 8
    x, a, b, w = _recall_layer(h_k, h_v, d)
    out = oracle.layer(x, a, b, w, np.zeros(h_v, np.float32), np.zeros(h_v, np.float32),
                       [0, d], h_k, h_v, d, d)
    v = x[:, 2 * h_k * d:].astype(np.float64)
    v = v * expit(v)                                   # SiLU of the v channels
    for h in range(h_v):
        vh = v[:, h * d:(h + 1) * d]
        # o_t = v_{t-1} / sqrt(d) for t >= 1; eps perturbs by <= 1e-6 relative
        np.testing.assert_allclose(out["o"][1:, h], vh[:-1] / np.sqrt(d), rtol=2e-6, atol=1e-9)


def test_varlen_sequences_do_not_leak():
    c = _layer_case(6, lengths=(5, 2, 9))
    keys = ("x", "a", "b", "conv_weight", "A_log", "dt_bias", "cu_seqlens")
    args = {kk: c[kk] for kk in keys}
    dims = (c["h_k"], c["h_v"], c["d_k"], c["d_v"])
    r1 = oracle.layer(*[args[kk] for kk in keys], *dims, window0=c["window0"], state0=c["state0"])
    x2 = c["x"].copy()
    x2[:5] += 3.0                                       # perturb sequence 0 only
    r2 = oracle.layer(x2, *[args[kk] for kk in keys[1:]], *dims, window0=c["window0"], state0=c["state0"])
    assert np.array_equal(r1["o"][5:], r2["o"][5:])
    assert np.array_equal(r1["state"][1:], r2["state"][1:])
    assert not np.allclose(r1["o"][:5], r2["o"][:5])


@pytest.mark.parametrize("T", [0, 1, 2, 3, 7])
def test_window_out_is_last_raw_inputs(T):
    c = _layer_case(8, lengths=(T,))
    r = oracle.layer(c["x"], c["a"], c["b"], c["conv_weight"], c["A_log"], c["dt_bias"],
                     c["cu_seqlens"], c["h_k"], c["h_v"], c["d_k"], c["d_v"],
                     window0=c["window0"], state0=c["state0"])
    hist = np.concatenate([c["window0"][0], c["x"]])
    np.testing.assert_array_equal(r["window"][0], hist[-3:].astype(np.float64))
    if T == 0:
        np.testing.assert_array_equal(r["state"][0], c["state0"][0].astype(np.float64))


def test_prefill_handoff_equals_one_long_prefill():
    """prefill(T1) -> (state, window) -> prefill(T2) == prefill(T1 + T2)."""
    c = _layer_case(10, lengths=(11,))
    kw = dict(h_k=c["h_k"], h_v=c["h_v"], d_k=c["d_k"], d_v=c["d_v"])
    p = (c["conv_weight"], c["A_log"], c["dt_bias"])
    full = oracle.layer(c["x"], c["a"], c["b"], *p, [0, 11], window0=c["window0"],
                        state0=c["state0"], **kw)
    first = oracle.layer(c["x"][:4], c["a"][:4], c["b"][:4], *p, [0, 4],
                         window0=c["window0"], state0=c["state0"], **kw)
    second = oracle.layer(c["x"][4:], c["a"][4:], c["b"][4:], *p, [0, 7],
                          window0=first["window"].astype(np.float32),
                          state0=first["state"].astype(np.float32), **kw)
    # the handoff rounds the state to float32 on the way; allow for that
    np.testing.assert_allclose(second["o"], full["o"][4:], rtol=0, atol=1e-6)
    np.testing.assert_allclose(second["state"], full["state"], rtol=0, atol=1e-6)
    np.testing.assert_array_equal(second["window"], full["window"])


def test_layer_matches_per_head_pipeline_and_threads_are_deterministic():
    """The layer equals front end + recurrence per (seq, head), its stored state
    is S transposed, and the thread count does not change a bit."""
    c = _layer_case(12, lengths=(6, 9))
    args = (c["x"], c["a"], c["b"], c["conv_weight"], c["A_log"], c["dt_bias"],
            c["cu_seqlens"], c["h_k"], c["h_v"], c["d_k"], c["d_v"])
    r1 = oracle.layer(*args, window0=c["window0"], state0=c["state0"], n_threads=1)
    r8 = oracle.layer(*args, window0=c["window0"], state0=c["state0"], n_threads=8)
    for kk in ("o", "state", "window"):
        assert np.array_equal(r1[kk], r8[kk])
    s, h = 1, 3
    lo, hi = 6, 15
    qh, kh, vv, g, be = oracle.frontend_head(
        c["x"][lo:hi], c["a"][lo:hi], c["b"][lo:hi], c["conv_weight"], c["A_log"],
        c["dt_bias"], c["h_k"], c["h_v"], c["d_k"], c["d_v"], h, window0=c["window0"][s])
    o_bf, S_bf = brute_force(qh[:8], kh[:8], vv[:8], g[:8], be[:8],
                             c["state0"][s, h].astype(np.float64).T)
    np.testing.assert_allclose(r1["o"][lo:lo + 8, h], o_bf, atol=1e-12)
    mask = np.zeros((2, c["h_v"]), bool)
    mask[s, h] = True
    rm = oracle.layer(*args, window0=c["window0"], state0=c["state0"], head_mask=mask)
    assert np.array_equal(rm["o"][lo:hi, h], r1["o"][lo:hi, h])
    assert np.array_equal(rm["state"][s, h], r1["state"][s, h])
    assert not rm["o"][lo:hi, h - 1].any()


# ---- gated RMSNorm of the output (the DeltaNet "gated norm") ------------------

def _norm_case(rows=5, d_v=32, seed=21):
    rng = np.random.default_rng(seed)
    o = rng.standard_normal((rows, d_v)).astype(np.float32)
    z = rng.standard_normal((rows, d_v)).astype(np.float32)
    w = rng.uniform(0.25, 2.0, d_v).astype(np.float32)
    return o, z, w


def test_gated_norm_closed_gate_is_zero():
    """SiLU(0) = 0: a zero gate gives a zero output whatever o and the weight."""
    o, z, w = _norm_case()
    assert not oracle.gated_rmsnorm(o, np.zeros_like(z), w).any()


def test_gated_norm_constant_row_closed_form():
    """A row of one value c has mean square c^2, so
    y_j = c / sqrt(c^2 + eps) * w_j * z_j * sigmoid(z_j)  (library sigmoid)."""
    _, z, w = _norm_case(rows=3)
    for c, eps in ((0.7, 1e-6), (-3.0, 0.0), (2e-3, 1e-6)):
        o = np.full_like(z, c)
        c = np.float64(np.float32(c))   # the value o actually holds
        ref = c / np.sqrt(c ** 2 + eps) * w.astype(np.float64) * \
            z.astype(np.float64) * expit(z.astype(np.float64))
        np.testing.assert_allclose(oracle.gated_rmsnorm(o, z, w, eps=eps), ref, rtol=1e-12,
                                   atol=1e-15)


def test_gated_norm_unit_rms_scale_invariance_and_weight_linearity():
    """With eps = 0, unit weight and an open gate (z = 40, SiLU(z) = 40 to
    1e-17), y / 40 has root mean square exactly 1; scaling o does not change y;
    y is linear in the weight, channel by channel, with no offset."""
    o, z, w = _norm_case()
    zo = np.full_like(z, 40.0)
    y = oracle.gated_rmsnorm(o, zo, np.ones_like(w), eps=0.0) / 40.0
    np.testing.assert_allclose(np.sqrt(np.mean(y ** 2, axis=-1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(oracle.gated_rmsnorm(4.0 * o, z, w, eps=0.0),
                               oracle.gated_rmsnorm(o, z, w, eps=0.0), rtol=1e-12)
    y1 = oracle.gated_rmsnorm(o, z, w)
    y2 = oracle.gated_rmsnorm(o, z, 2.0 * w)
    np.testing.assert_allclose(y2, 2.0 * y1, rtol=1e-12)


# ---------------------------------------------------------------- decay / beta projection

def test_gate_projection_worked_example():
    """A 2-token, 3-wide hidden state and h_v = 2 (four weight rows: two decay
    rows, then two beta rows), worked out by hand from the definition
    a[t][h] = sum_i hidden[t][i] W[h][i], b[t][h] = sum_i hidden[t][i] W[2 + h][i]."""
    hidden = np.array([[1.0, 2.0, 3.0],
                       [-1.0, 0.5, 4.0]])
    w = np.array([[1.0, 0.0, 0.0],     # a, head 0: the first channel
                  [0.0, 1.0, -1.0],    # a, head 1: second minus third
                  [2.0, 2.0, 2.0],     # b, head 0: twice the sum
                  [0.0, 0.0, 0.25]])   # b, head 1: a quarter of the third
    a, b = oracle.gate_projection(hidden, w, 2)
    np.testing.assert_array_equal(a, [[1.0, -1.0], [-1.0, -3.5]])
    np.testing.assert_array_equal(b, [[12.0, 0.75], [7.0, 1.0]])


def test_gate_projection_unit_rows_select_channels():
    """Weight rows that are unit vectors e_{p(r)} pick channel p(r) of every
    token exactly: decay rows the first h_v picks, beta rows the rest."""
    rng = RNG(51)
    n, d_model, h_v = 37, 96, 8
    hidden = rng.standard_normal((n, d_model)).astype(np.float32)
    pick = rng.permutation(d_model)[:2 * h_v]
    w = np.zeros((2 * h_v, d_model), np.float32)
    w[np.arange(2 * h_v), pick] = 1.0
    a, b = oracle.gate_projection(hidden, w, h_v)
    np.testing.assert_array_equal(a, hidden[:, pick[:h_v]].astype(np.float64))
    np.testing.assert_array_equal(b, hidden[:, pick[h_v:]].astype(np.float64))


def test_gate_projection_linear_in_both_operands():
    """Additive in the hidden state and in the weights, token by token: the
    projection of a sum is the sum of the projections (to float64 rounding),
    and a token's outputs depend on that token's row only."""
    rng = RNG(52)
    n, d_model, h_v = 19, 160, 4
    # multiples of 1/8 below 64 in magnitude: every input and every sum of two
    # is exact in the single precision the oracle takes its inputs in
    h1, h2 = (rng.integers(-511, 512, (n, d_model)) / 8.0 for _ in range(2))
    w1, w2 = (rng.integers(-511, 512, (2 * h_v, d_model)) / 8.0 for _ in range(2))
    a12, b12 = oracle.gate_projection(h1 + h2, w1, h_v)
    a1, b1 = oracle.gate_projection(h1, w1, h_v)
    a2, b2 = oracle.gate_projection(h2, w1, h_v)
    scale = np.abs(np.concatenate([a1, a2, b1, b2])).max()
    np.testing.assert_allclose(a12, a1 + a2, atol=1e-12 * scale * d_model)
    np.testing.assert_allclose(b12, b1 + b2, atol=1e-12 * scale * d_model)
    aw, bw = oracle.gate_projection(h1, w1 + w2, h_v)
    a3, b3 = oracle.gate_projection(h1, w2, h_v)
    np.testing.assert_allclose(aw, a1 + a3, atol=1e-12 * scale * d_model)
    np.testing.assert_allclose(bw, b1 + b3, atol=1e-12 * scale * d_model)
    hz = h1.copy()
    hz[5] = 0.0
    az, bz = oracle.gate_projection(hz, w1, h_v)
    assert not az[5].any() and not bz[5].any()
    keep = np.arange(n) != 5
    np.testing.assert_array_equal(az[keep], a1[keep])
    np.testing.assert_array_equal(bz[keep], b1[keep])


# ---------------------------------------------------------------- slots and checkpoints

def test_slot_copy_moves_exactly_the_named_slots():
    rng = RNG(41)
    st = rng.standard_normal((6, 2, 3, 4))
    cw = rng.standard_normal((6, 3, 5))
    st2, cw2 = oracle.slot_copy(st, cw, [4, -1, 0], [1, 3, 5])
    np.testing.assert_array_equal(st2[1], st[4])
    np.testing.assert_array_equal(cw2[1], cw[4])
    np.testing.assert_array_equal(st2[5], st[0])
    for s_ in (0, 2, 3, 4):                      # sources and untouched slots (3: padding pair)
        np.testing.assert_array_equal(st2[s_], st[s_])
        np.testing.assert_array_equal(cw2[s_], cw[s_])
    # snapshot then restore gives back the original slot after it was overwritten
    snap_st, snap_cw = oracle.slot_copy(st, cw, [2], [5])
    snap_st[2] += 1.0
    back_st, back_cw = oracle.slot_copy(snap_st, snap_cw, [5], [2])
    np.testing.assert_array_equal(back_st[2], st[2])
    np.testing.assert_array_equal(back_cw[2], cw[2])


@pytest.mark.parametrize("lengths,every", [((13,), 4), ((16, 5, 9), 4), ((7,), 8), ((24,), 8)])
def test_checkpoints_count_and_resume(lengths, every):
    """There are ceil(len / every) - 1 checkpoints per sequence, and resuming
    from checkpoint k over the remaining tokens reproduces the full run's
    outputs for them and its final state and window -- a checkpoint one token
    off would apply that token twice or not at all."""
    c = _layer_case(50 + every, lengths=lengths)
    kw = dict(h_k=c["h_k"], h_v=c["h_v"], d_k=c["d_k"], d_v=c["d_v"])
    p = (c["conv_weight"], c["A_log"], c["dt_bias"])
    full = oracle.layer(c["x"], c["a"], c["b"], *p, c["cu_seqlens"], window0=c["window0"],
                        state0=c["state0"], **kw)
    ck = oracle.prefill_checkpoints(c["x"], c["a"], c["b"], *p, c["cu_seqlens"], every=every,
                                    window0=c["window0"], state0=c["state0"], **kw)
    cu = c["cu_seqlens"]
    for bi, (states, windows) in enumerate(ck):
        s0, ln = int(cu[bi]), int(cu[bi + 1] - cu[bi])
        assert states.shape[0] == windows.shape[0] == -(-ln // every) - 1
        for k in range(1, states.shape[0] + 1):
            t = k * every
            rest = oracle.layer(c["x"][s0 + t:s0 + ln], c["a"][s0 + t:s0 + ln],
                                c["b"][s0 + t:s0 + ln], *p, [0, ln - t],
                                window0=windows[k - 1:k].astype(np.float32),
                                state0=states[k - 1:k].astype(np.float32), **kw)
            # the resume rounds the state to float32 on the way; allow for that
            np.testing.assert_allclose(rest["o"], full["o"][s0 + t:s0 + ln], rtol=0, atol=1e-6)
            np.testing.assert_allclose(rest["state"][0], full["state"][bi], rtol=0, atol=1e-6)
            np.testing.assert_array_equal(rest["window"][0], full["window"][bi])
            # the window of checkpoint k is the raw inputs just before position t
            np.testing.assert_array_equal(windows[k - 1], c["x"][s0 + t - 3:s0 + t])
