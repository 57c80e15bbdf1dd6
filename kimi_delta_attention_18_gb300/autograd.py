"""The prefill as a differentiable PyTorch operation: the forward is
kda_prefill_chunked, the backward kda_prefill_backward (both libkda kernels).

``kda_prefill(q, k, v, g, beta, S0=None, cu_seqlens=None)`` returns
``(o, S_final)``; gradients flow to q, k, v, g (the log-decay), beta and S0 for
any loss of o and S_final.  The library's gradients are fp32; they are cast to
each input's dtype (BF16 q, k, v get BF16 gradients).
"""
from __future__ import annotations

import torch

from . import _native as _k


class KDAPrefill(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, S0, cu_seqlens, num_segments):
        out, S_final = _k.prefill_chunked(q, k, v, g, beta, S0, cu_seqlens,
                                          num_segments=num_segments)
        ctx.save_for_backward(q, k, v, g, beta, S0, cu_seqlens)
        ctx.has_S0 = S0 is not None
        return out, S_final

    @staticmethod
    def backward(ctx, d_out, d_S_final):
        q, k, v, g, beta, S0, cu_seqlens = ctx.saved_tensors
        if d_out is None:
            d_out = torch.zeros((q.shape[0], q.shape[1], v.shape[2]), dtype=q.dtype,
                                device=q.device)
        d_out = d_out.to(q.dtype).contiguous()
        if d_S_final is not None:
            d_S_final = d_S_final.float().contiguous()
        dq, dk, dv, dg, dbeta, dS0 = _k.prefill_backward(q, k, v, g, beta, S0, cu_seqlens, d_out,
                                                         d_S_final, want_dS0=ctx.has_S0)
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), dg, dbeta,
                dS0 if ctx.has_S0 else None, None, None)


def kda_prefill(q, k, v, g, beta, S0=None, cu_seqlens=None, *, num_segments=0):
    """Differentiable one-call prefill (see the module docstring).  Inputs as for
    ``prefill_chunked``; returns ``(o, S_final)``."""
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, q.shape[0]], dtype=torch.int32, device=q.device)
    return KDAPrefill.apply(q, k, v, g, beta, S0, cu_seqlens, num_segments)
