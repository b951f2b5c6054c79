"""Independent float64 evaluations used to pin the oracle (numpy only).

Neither function shares code with the oracle (C, token-by-token loops) nor with
the CUDA library.  Both work in the math convention S in R^{d_v x d_k}, o = S q.

brute_force:  the unrolled closed form of the gated delta rule,
    S_t = S_0 M_1 ... M_t + sum_{s<=t} beta_s v_s k_s^T M_{s+1} ... M_t,
    M_r = exp(g_r) (I - beta_r k_r k_r^T),
  evaluated with explicit d_k x d_k matrix products for every t (O(T^2)
  products, so only for T <= 8).

chunked_wy:  the chunked form the GPU prefill uses (Gated DeltaNet's chunkwise
  WY representation): inside a chunk of C tokens with cumulative log-decay
  gamma, A = strict_tril(diag(beta) K K^T * exp(gamma_r - gamma_s)),
  T = (I + A)^-1, U = T diag(beta) V, Wk = T diag(beta exp(gamma)) K,
  W = U - Wk S^T, O = diag(exp(gamma)) Q S^T + tril(Q K^T * exp(gamma_r -
  gamma_s)) W, S <- exp(gamma_C) S + W^T diag(exp(gamma_C - gamma)) K.
  The inverse is taken with numpy's general solver (no special structure).
"""
from __future__ import annotations

import numpy as np


def brute_force(q, k, v, g, beta, S0=None):
    T, d_k = k.shape
    d_v = v.shape[1]
    S0 = np.zeros((d_v, d_k)) if S0 is None else np.asarray(S0, np.float64)
    eye = np.eye(d_k)
    M = [np.exp(g[r]) * (eye - beta[r] * np.outer(k[r], k[r])) for r in range(T)]

    def prod(lo, hi):  # M_lo ... M_hi (inclusive); identity if empty
        out = eye.copy()
        for r in range(lo, hi + 1):
            out = out @ M[r]
        return out

    o = np.zeros((T, d_v))
    S_t = S0
    for t in range(T):
        S_t = S0 @ prod(0, t)
        for s in range(t + 1):
            S_t = S_t + beta[s] * np.outer(v[s], k[s]) @ prod(s + 1, t)
        o[t] = S_t @ q[t]
    return o, S_t


def chunk_inverse(k, g, beta):
    """(I + strict_tril(diag(beta) K K^T * exp(gamma_r - gamma_s)))^-1 for one chunk."""
    C = k.shape[0]
    gam = np.cumsum(g)
    A = np.tril(beta[:, None] * (k @ k.T) * np.exp(gam[:, None] - gam[None, :]), -1)
    return np.linalg.solve(np.eye(C) + A, np.eye(C))


def chunked_wy(q, k, v, g, beta, S0=None, C=16):
    T, d_k = k.shape
    d_v = v.shape[1]
    S = np.zeros((d_v, d_k)) if S0 is None else np.array(S0, np.float64)
    o = np.zeros((T, d_v))
    for c0 in range(0, T, C):
        c1 = min(c0 + C, T)
        qc, kc, vc, gc, bc = q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1]
        gam = np.cumsum(gc)
        Tinv = chunk_inverse(kc, gc, bc)
        U = Tinv @ (bc[:, None] * vc)
        Wk = Tinv @ ((bc * np.exp(gam))[:, None] * kc)
        W = U - Wk @ S.T
        P = np.tril((qc @ kc.T) * np.exp(gam[:, None] - gam[None, :]))
        o[c0:c1] = np.exp(gam)[:, None] * (qc @ S.T) + P @ W
        S = np.exp(gam[-1]) * S + W.T @ (np.exp(gam[-1] - gam)[:, None] * kc)
    return o, S
