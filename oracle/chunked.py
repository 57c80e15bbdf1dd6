"""Chunked (WY / UT-transform) form of the KDA recurrence, fp64 numpy.

TEST INFRASTRUCTURE ONLY: a second, independent way of computing what
``oracle.kda_forward`` computes, used by the self-checks to pin the algebra that
a chunked implementation relies on.  It is never the reference the GPU path is
compared with (that is the token-by-token oracle).

The chunk size is free (the pages use 16-token blocks so that the in-block
exponent factors stay inside BF16 range: Kimi K3 technical-report digest,
section 2.1 (1)); in exact arithmetic the result does not depend on it.

For one head and one chunk of C tokens starting from state S (dk x dv), with
Gamma_r = g_1 + ... + g_r (per key channel) and P_r = Diag(exp(Gamma_r)):

    Kh = K * exp(Gamma)         (row r scaled by exp(Gamma_r))
    Kt = K * exp(-Gamma)
    Qh = Q * exp(Gamma)
    Kb = K * exp(Gamma_C - Gamma)
    L  = strictly lower part of Kh Kt^T       L[r,i] = sum_c k_rc k_ic e^{Gamma_rc - Gamma_ic}
    Mq = lower part (with diagonal) of Qh Kt^T
    T  = (I + Diag(beta) L)^{-1} Diag(beta)
    W  = T Kh,   Ut = T V
    U  = Ut - W S                 (the per-token "write differences")
    O  = Qh S + Mq U
    S' = P_C S + Kb^T U

U's row r equals beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r), the difference
the delta rule writes; the rest follows by unrolling decay, erase and write.
"""
from __future__ import annotations

import numpy as np


def chunk_step(S, q, k, v, g, beta):
    """One chunk for one head. q, k, g: [C, dk]; v: [C, dv]; beta: [C]; S: [dk, dv].
    Returns (O [C, dv], S_next [dk, dv])."""
    C = k.shape[0]
    Gam = np.cumsum(g, axis=0)
    Kh = k * np.exp(Gam)
    Kt = k * np.exp(-Gam)
    Qh = q * np.exp(Gam)
    Kb = k * np.exp(Gam[-1][None, :] - Gam)
    L = np.tril(Kh @ Kt.T, -1)
    Mq = np.tril(Qh @ Kt.T, 0)
    T = np.linalg.solve(np.eye(C) + beta[:, None] * L, np.diag(beta))
    W = T @ Kh
    Ut = T @ v
    U = Ut - W @ S
    O = Qh @ S + Mq @ U
    S_next = np.exp(Gam[-1])[:, None] * S + Kb.T @ U
    return O, S_next


def kda_forward_chunked(q, k, v, g, beta, S0=None, cu_seqlens=None, chunk=16):
    """Same contract as ``oracle.kda_forward`` (fp64), computed chunk by chunk;
    the last chunk of each sequence may be partial."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, np.int64)
    N = len(cu) - 1
    out = np.zeros((T, H, dv))
    SF = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], np.float64)
            for t0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                t1 = min(t0 + chunk, int(cu[n + 1]))
                O, S = chunk_step(S, q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h],
                                  beta[t0:t1, h])
                out[t0:t1, h] = O
            SF[n, h] = S
    return out, SF
