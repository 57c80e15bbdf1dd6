"""Context parallelism of the prefill across ranks (KCP, "Kimi K3 Architecture
Explained" / the technical-report digest, section 2.4 (1)).

Every sequence is split into W segments, one per rank (the chunk-aligned split of
kda_state_transfer).  The state after a segment is linear in the state before it,
S_after = A_s S_before + B_s, so rank r computes only its segment's transfer matrix
A_r and zero-start state B_r, the ranks exchange these pairs with one all-gather
(their size, N * H * (dk * dk + dk * dv) fp32, does not depend on the sequence
length), every rank scans the W pairs locally for its segment's start state, and
reruns its segment from it.  Every rank also gets S_final.

The compute is libkda's (kda_state_transfer, kda_state_compose,
kda_prefill_segments); this module is the exchange around it.  Every rank is
given the whole packed batch (the kernels read only the rank's segment of it);
rank r returns outputs for its segment's tokens and zeros elsewhere.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch

from . import _native as _k


@dataclass
class KCPOps:
    """The three compute steps.  The defaults are the libkda entry points.

    transfer(k, v, g, beta, cu_seqlens, W, r) -> (A_r [N,H,dk,dk], B_r [N,H,dk,dv])
    compose(A [U,W,dk,dk], B [U,W,dk,dv], S0 [U,dk,dv] or None) -> (starts [U,W,dk,dv], S_final [U,dk,dv])
    segment(q, k, v, g, beta, starts [N,H,W,dk,dv], cu_seqlens, W, r) -> out [T,H,dv]
    """
    transfer: Callable
    compose: Callable
    segment: Callable


def _transfer(k, v, g, beta, cu_seqlens, W, r):
    A, B = _k.state_transfer(k, v, g, beta, cu_seqlens, W, seg_begin=r, seg_end=r + 1)
    return A[:, :, r].contiguous(), B[:, :, r].contiguous()


def _compose(A, B, S0):
    return _k.state_compose(A, B, S0)


def _segment(q, k, v, g, beta, starts, cu_seqlens, W, r):
    out = torch.zeros((q.shape[0], q.shape[1], v.shape[2]), dtype=q.dtype, device=q.device)
    _k.prefill_segments(q, k, v, g, beta, starts, cu_seqlens, W, seg_begin=r, seg_end=r + 1,
                        out=out, want_final_state=False)
    return out


LIBKDA_OPS = KCPOps(_transfer, _compose, _segment)


def local_pairs(k, v, g, beta, cu_seqlens, W, r, ops=None):
    """Rank r's (A_r, B_r): the transfer matrix and zero-start state of segment r
    of every (sequence, head)."""
    ops = ops or LIBKDA_OPS
    return ops.transfer(k, v, g, beta, cu_seqlens, W, r)


def finish(q, k, v, g, beta, S0, cu_seqlens, W, r, A_all, B_all, ops=None):
    """Given every rank's pairs (A_all [N,H,W,dk,dk], B_all [N,H,W,dk,dv]), scan
    them for the segment start states and run segment r from its start state.
    Returns (out with segment r's tokens filled, S_final [N,H,dk,dv])."""
    ops = ops or LIBKDA_OPS
    N, H, _, dk, dv = B_all.shape
    U = N * H
    S0u = None if S0 is None else S0.reshape(U, dk, dv)
    starts, S_final = ops.compose(A_all.reshape(U, W, dk, dk), B_all.reshape(U, W, dk, dv), S0u)
    out = ops.segment(q, k, v, g, beta, starts.reshape(N, H, W, dk, dv), cu_seqlens, W, r)
    return out, S_final.reshape(N, H, dk, dv)


def kcp_prefill(q, k, v, g, beta, S0, cu_seqlens, *, group=None, ops=None):
    """The prefill of the whole batch split over the ranks of ``group`` (one
    segment of every sequence per rank), with one all-gather of the fixed-size
    (A, B) pairs.  Returns (out, S_final): out holds this rank's segment's
    outputs (zeros at other ranks' tokens), S_final the final states (the same on
    every rank)."""
    import torch.distributed as dist
    W = dist.get_world_size(group)
    r = dist.get_rank(group)
    A_r, B_r = local_pairs(k, v, g, beta, cu_seqlens, W, r, ops)
    A_parts = [torch.empty_like(A_r) for _ in range(W)]
    B_parts = [torch.empty_like(B_r) for _ in range(W)]
    dist.all_gather(A_parts, A_r, group=group)
    dist.all_gather(B_parts, B_r, group=group)
    A_all = torch.stack(A_parts, dim=2)
    B_all = torch.stack(B_parts, dim=2)
    return finish(q, k, v, g, beta, S0, cu_seqlens, W, r, A_all, B_all, ops)


def segment_token_mask(cu_seqlens, W, r, T):
    """Bool [T]: the tokens of segment r (of W) of every sequence, the tokens rank r
    outputs (the chunk-aligned split of kda_state_transfer)."""
    cu = [int(c) for c in torch.as_tensor(cu_seqlens).cpu().tolist()]
    mask = torch.zeros(T, dtype=torch.bool)
    for n in range(len(cu) - 1):
        L = cu[n + 1] - cu[n]
        c = -(-L // 16)
        a = cu[n] + min(L, (r * c) // W * 16)
        b = cu[n] + min(L, ((r + 1) * c) // W * 16)
        mask[a:b] = True
    return mask
