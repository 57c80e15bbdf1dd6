"""KDA oracle: plain fp64 CPU implementation of the Kimi Delta Attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library never loads it and shares no code with it.

Contents
--------
``kda_forward``         token-by-token recurrence (C, ``kda_oracle.c``) over
                        packed variable-length sequences; returns outputs and
                        final states.  Follows "Kimi K3 Architecture Explained",
                        section 3 (decay, then erase, then write) and the Kimi K3
                        technical-report digest, section 2.1 (1) (delta rule
                        with a channel-wise forget gate, g_min = -5).
``kda_decode_step``     one token per sequence: the same recurrence with T = 1.
``segment_bounds``      the context-parallel split of each sequence into
                        chunk-aligned segments (digest section 2.4 (1), KCP).
``kda_state_transfer``  per segment, the transfer matrix A (the recurrence run
                        from the identity with zero values) and the
                        zero-initial state B (the recurrence run from zeros):
                        S_end = A S_start + B (digest section 2.4 (1)).
``kda_state_compose``   the prefix scan S_s = A_{s-1} S_{s-1} + B_{s-1}.
``kda_backward``        gradients of the recurrence for <d_out, o> + <d_S_final,
                        S_final> with respect to q, k, v, g, beta and S0 (fp64
                        PyTorch autograd over the token loop; small problems).
``gate_prologue``       the inputs from their pre-activations: g = -5 sigmoid(x_g)
                        (digest section 2.1 (1)), beta = sigmoid(x_beta), and q, k
                        divided by their L2 norm per (token, head), as the input
                        recipe prepares them (a zero row stays zero).

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
closed forms, brute-force matrix products, special cases and invariants; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libkda_oracle.so`` (gcc, fp64, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        f = lib.kda_oracle_forward
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int] + \
            [ctypes.c_void_p] * 8 + [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _lib = lib
    return _lib


def host_threads() -> int:
    """Worker threads the oracle uses by default: the cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def kda_forward(q, k, v, g, beta, S0=None, cu_seqlens=None, *, erase=True,
                with_output=True, threads=None, col_block=None):
    """Token-by-token KDA in fp64.

    Shapes (packed over sequences): q, k, g ``[T, H, dk]``; v ``[T, H, dv]``;
    beta ``[T, H]``; S0 ``[N, H, dk, dv]`` or None (zeros); cu_seqlens ``[N+1]``
    or None (one sequence of length T).  Returns ``(out [T,H,dv] or None,
    S_final [N,H,dk,dv])`` as fp64 numpy arrays.  ``erase=False`` drops only the
    erase step (the gated-linear-attention reading used by the self-checks).
    """
    k = _f64(k); v = _f64(v); g = _f64(g); beta = _f64(beta)
    q = _f64(q) if q is not None else None
    T, H, dk = k.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0), "bad cu_seqlens"
    assert g.shape == (T, H, dk) and beta.shape == (T, H) and v.shape[:2] == (T, H)
    S0a = None if S0 is None else _f64(S0).reshape(N, H, dk, dv)
    out = np.zeros((T, H, dv)) if with_output else None
    SF = np.zeros((N, H, dk, dv))
    if threads is None:
        threads = host_threads()
    if col_block is None:
        # enough jobs to keep every thread busy, never below 8 columns per job
        units = max(1, N * H)
        per = max(1, -(-threads // units))
        col_block = max(8, -(-dv // per)) if per > 1 else dv
    rc = _load().kda_oracle_forward(
        N, cu.ctypes.data, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(S0a), _ptr(out), SF.ctypes.data, 1 if erase else 0, int(col_block), int(threads))
    if rc != 0:
        raise ValueError("kda_oracle_forward rejected its arguments")
    return out, SF


def kda_decode_step(q, k, v, g, beta, S, *, threads=None):
    """One decode token per sequence: shapes ``[B, H, d]``, beta ``[B, H]``,
    S ``[B, H, dk, dv]``.  Returns ``(out [B,H,dv], S_new [B,H,dk,dv])``."""
    B = np.asarray(k).shape[0]
    cu = np.arange(B + 1, dtype=np.int64)
    return kda_forward(q, k, v, g, beta, S0=S, cu_seqlens=cu, threads=threads)


def segment_bounds(cu_seqlens, num_segments: int, chunk: int = 16):
    """Split each sequence into ``num_segments`` contiguous, chunk-aligned pieces.

    Sequence n has c_n = ceil(len_n / chunk) chunks; segment s takes chunks
    [floor(s c_n / S), floor((s+1) c_n / S)), clipped to the sequence end.
    Returns an int64 array ``[N, S, 2]`` of absolute token ranges.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    Sg = int(num_segments)
    out = np.zeros((N, Sg, 2), dtype=np.int64)
    for n in range(N):
        L = int(cu[n + 1] - cu[n])
        c = -(-L // chunk)
        for s in range(Sg):
            c0 = (s * c) // Sg
            c1 = ((s + 1) * c) // Sg
            out[n, s, 0] = cu[n] + min(L, c0 * chunk)
            out[n, s, 1] = cu[n] + min(L, c1 * chunk)
    return out


def _segments_as_sequences(bounds):
    """Segments are contiguous token ranges, so a flat list of them is itself a
    valid packing when run over a copy of the tokens gathered in order."""
    N, Sg, _ = bounds.shape
    idx, cu = [], [0]
    for n in range(N):
        for s in range(Sg):
            a, b = int(bounds[n, s, 0]), int(bounds[n, s, 1])
            idx.append(np.arange(a, b, dtype=np.int64))
            cu.append(cu[-1] + (b - a))
    return np.concatenate(idx) if idx else np.zeros(0, np.int64), np.asarray(cu, np.int64)


def kda_state_transfer(k, v, g, beta, cu_seqlens, num_segments, *, chunk=16, threads=None):
    """Per (sequence, head, segment): transfer matrix A [dk, dk] and zero-initial
    state B [dk, dv] such that the state after the segment is A S_start + B.

    A is the recurrence run from S = I with zero values; B the recurrence run
    from S = 0 with the segment's values (Kimi K3 technical-report digest,
    section 2.4 (1): the recurrent state split into a transfer matrix and a
    zero-initial state).  Returns ``(A [N,H,S,dk,dk], B [N,H,S,dk,dv])``.
    """
    k = _f64(k); v = _f64(v); g = _f64(g); beta = _f64(beta)
    T, H, dk = k.shape
    dv = v.shape[2]
    bounds = segment_bounds(cu_seqlens, num_segments, chunk)
    N, Sg, _ = bounds.shape
    idx, cu = _segments_as_sequences(bounds)
    ks, vs, gs, bs = k[idx], v[idx], g[idx], beta[idx]
    M = N * Sg
    eye = np.broadcast_to(np.eye(dk), (M, H, dk, dk))
    _, A = kda_forward(None, ks, np.zeros((len(idx), H, dk)), gs, bs, S0=eye, cu_seqlens=cu,
                       with_output=False, threads=threads)
    _, B = kda_forward(None, ks, vs, gs, bs, S0=None, cu_seqlens=cu, with_output=False,
                       threads=threads)
    A = A.reshape(N, Sg, H, dk, dk).transpose(0, 2, 1, 3, 4).copy()
    B = B.reshape(N, Sg, H, dk, dv).transpose(0, 2, 1, 3, 4).copy()
    return A, B


def kda_state_compose(A, B, S0=None):
    """Prefix scan over segments: start_0 = S0 (or zeros),
    start_s = A_{s-1} start_{s-1} + B_{s-1}; returns ``(starts [U,S,dk,dv],
    S_final [U,dk,dv])`` for A ``[U,S,dk,dk]``, B ``[U,S,dk,dv]``."""
    A = _f64(A); B = _f64(B)
    U, Sg, dk, dv = B.shape
    cur = np.zeros((U, dk, dv)) if S0 is None else _f64(S0).reshape(U, dk, dv).copy()
    starts = np.zeros((U, Sg, dk, dv))
    for s in range(Sg):
        starts[:, s] = cur
        cur = np.matmul(A[:, s], cur) + B[:, s]
    return starts, cur


def gate_prologue(q, k, x_g, x_beta):
    """Fused-prologue reference, in fp64: returns (q / |q|, k / |k|, g, beta) with
    g = -5 sigmoid(x_g) (the bounded gate of the digest, section 2.1 (1): g in
    (-5, 0)) and beta = sigmoid(x_beta); norms over the last (key-channel) axis
    per (token, head); a row of zeros stays zero."""
    q, k, x_g, x_beta = _f64(q), _f64(k), _f64(x_g), _f64(x_beta)

    def unit(x):
        n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
        return np.where(n > 0, x / np.where(n > 0, n, 1.0), 0.0)

    sig = lambda z: 1.0 / (1.0 + np.exp(-z))
    return unit(q), unit(k), -5.0 * sig(x_g), sig(x_beta)


def kda_backward(q, k, v, g, beta, S0, cu_seqlens, d_out, d_S_final=None):
    """Gradients of the recurrence (the same token loop as ``kda_forward``: decay,
    erase, write, then read o_t = S_t^T q_t; "Kimi K3 Architecture Explained",
    section 3) with respect to q, k, v, g, beta and S0, for the loss
    <d_out, o> + <d_S_final, S_final>.  Plain fp64 PyTorch on the CPU: the forward
    written out token by token and differentiated by autograd (a library
    primitive); small problems only.  Returns (dq, dk, dv, dg, dbeta, dS0) as numpy
    arrays (dS0 zero-shaped like S0, or None when S0 is None)."""
    import torch

    t = lambda a: torch.tensor(_f64(a), dtype=torch.float64, requires_grad=True)
    Q, K, V, G, B = t(q), t(k), t(v), t(g), t(beta)
    T, H, dk = Q.shape
    dv = V.shape[2]
    cu = [int(c) for c in np.asarray(cu_seqlens)]
    N = len(cu) - 1
    S0t = t(S0) if S0 is not None else None
    outs, finals = [], []
    for n in range(N):
        rows = []
        fin = []
        for h in range(H):
            S = S0t[n, h] if S0t is not None else torch.zeros(dk, dv, dtype=torch.float64)
            o_h = []
            for i in range(cu[n], cu[n + 1]):
                S = torch.exp(G[i, h])[:, None] * S                      # decay
                kk = K[i, h]
                S = S - B[i, h] * torch.outer(kk, kk @ S)                # erase
                S = S + B[i, h] * torch.outer(kk, V[i, h])               # write
                o_h.append(S.T @ Q[i, h])                                # read
            rows.append(torch.stack(o_h) if o_h else torch.zeros(0, dv, dtype=torch.float64))
            fin.append(S)
        outs.append(torch.stack(rows, dim=1))
        finals.append(torch.stack(fin))
    O = torch.cat(outs, dim=0)
    SF = torch.stack(finals)
    loss = (O * torch.tensor(_f64(d_out))).sum()
    if d_S_final is not None:
        loss = loss + (SF * torch.tensor(_f64(d_S_final))).sum()
    loss.backward()
    g_or_zero = lambda x: (x.grad if x.grad is not None else torch.zeros_like(x)).numpy()
    dS0 = g_or_zero(S0t) if S0t is not None else None
    return g_or_zero(Q), g_or_zero(K), g_or_zero(V), g_or_zero(G), g_or_zero(B), dS0
