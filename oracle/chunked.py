"""Chunked (WY / UT-transform) form of the KDA recurrence, fp64 numpy.

TEST INFRASTRUCTURE ONLY: a second, independent way of computing what
``oracle.kda_forward`` and ``oracle.kda_backward`` compute, used by the
self-checks to pin the algebra that a chunked implementation relies on (forward
and adjoint).  It is never the reference the GPU path is compared with (that is
the token-by-token oracle).

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


def chunk_step_backward(S, q, k, v, g, beta, dO, dS_next):
    """Adjoint of ``chunk_step`` for one head and one chunk: given the chunk's start
    state S and the adjoints dO [C, dv] of its outputs and dS_next [dk, dv] of its
    end state, returns (dS, dq, dk, dv, dg, dbeta) — the same gradients the
    token-by-token recurrence gives, through the chunked form's own algebra:

        dU  = Mq^T dO + Kb dS'                   R = V - Kh S,  U = T R
        dT  = dU R^T,  dR = T^T dU,  dV = dR
        T = Y Diag(beta), Y = (I + Diag(beta) L)^{-1}:
            dbeta_j += sum_i dT_ij Y_ij,   dMb = -Y^T (dT Diag(beta)) Y^T,
            dbeta_i += sum_j dMb_ij L_ij,   dL = Diag(beta) dMb (strictly lower)
        dMq = lower(dO U^T);  Kh, Kt, Qh, Kb, e^{Gamma_C} -> K, Q, Gamma;
        dg = reverse cumulative sum of dGamma over the chunk.
    """
    C = k.shape[0]
    Gam = np.cumsum(g, axis=0)
    Ep, Em = np.exp(Gam), np.exp(-Gam)
    Eb = np.exp(Gam[-1][None, :] - Gam)
    eC = np.exp(Gam[-1])
    Kh, Kt, Qh, Kb = k * Ep, k * Em, q * Ep, k * Eb
    L = np.tril(Kh @ Kt.T, -1)
    Mq = np.tril(Qh @ Kt.T, 0)
    Y = np.linalg.inv(np.eye(C) + beta[:, None] * L)
    T = Y * beta[None, :]
    R = v - Kh @ S
    U = T @ R
    # O = Qh S + Mq U,  S' = Diag(eC) S + Kb^T U
    dU = Mq.T @ dO + Kb @ dS_next
    dS = Qh.T @ dO + eC[:, None] * dS_next
    dQh = dO @ S.T
    dMq = np.tril(dO @ U.T, 0)
    dKb = U @ dS_next.T
    deC = np.sum(dS_next * S, axis=1)
    # U = T R, R = V - Kh S
    dT = dU @ R.T
    dR = T.T @ dU
    dv_ = dR
    dKh = -dR @ S.T
    dS = dS - Kh.T @ dR
    # T = Y Diag(beta), Y = (I + Diag(beta) L)^{-1}
    dbeta = np.sum(dT * Y, axis=0)
    dMb = -Y.T @ (dT * beta[None, :]) @ Y.T
    dbeta = dbeta + np.sum(dMb * L, axis=1)
    dL = np.tril(beta[:, None] * dMb, -1)
    # L = strict_lower(Kh Kt^T), Mq = lower(Qh Kt^T)
    dKh = dKh + dL @ Kt
    dKt = dL.T @ Kh + dMq.T @ Qh
    dQh = dQh + dMq @ Kt
    # to K, Q and Gamma
    dk_ = dKh * Ep + dKt * Em + dKb * Eb
    dq_ = dQh * Ep
    dGam = dKh * Kh - dKt * Kt + dQh * Qh - dKb * Kb
    dGam[-1] += np.sum(dKb * Kb, axis=0) + deC * eC
    dg_ = np.cumsum(dGam[::-1], axis=0)[::-1]
    return dS, dq_, dk_, dv_, dg_, dbeta


def kda_backward_chunked(q, k, v, g, beta, S0, cu_seqlens, d_out, d_S_final=None, chunk=16):
    """Same contract as ``oracle.kda_backward`` (fp64), computed chunk by chunk: a
    forward pass keeping each chunk's start state, then ``chunk_step_backward``
    from the last chunk to the first."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64); d_out = np.asarray(d_out, np.float64)
    T, H, dk = k.shape
    dv = v.shape[2]
    cu = np.asarray(cu_seqlens, np.int64)
    N = len(cu) - 1
    grads = [np.zeros((T, H, dk)), np.zeros((T, H, dk)), np.zeros((T, H, dv)),
             np.zeros((T, H, dk)), np.zeros((T, H))]
    dS0 = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], np.float64)
            spans, starts = [], []
            for t0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                t1 = min(t0 + chunk, int(cu[n + 1]))
                spans.append((t0, t1))
                starts.append(S)
                _, S = chunk_step(S, q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h],
                                  beta[t0:t1, h])
            dS = np.zeros((dk, dv)) if d_S_final is None else np.array(d_S_final[n, h])
            for (t0, t1), Sc in zip(spans[::-1], starts[::-1]):
                dS, dq_, dk_, dv_, dg_, db_ = chunk_step_backward(
                    Sc, q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h], beta[t0:t1, h],
                    d_out[t0:t1, h], dS)
                for arr, val in zip(grads, (dq_, dk_, dv_, dg_, db_)):
                    arr[t0:t1, h] = val
            dS0[n, h] = dS
    return (*grads, dS0)
