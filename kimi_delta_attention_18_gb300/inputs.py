"""Seeded synthetic inputs for the KDA path.

This module draws inputs only; it holds none of the recurrence's arithmetic and is
the one module the CUDA path's tests and the oracle both consume.

Recipe (every workload): q, k ~ N(0, 1), each L2-normalised per (token, head) in
fp32 and then cast to the activation dtype; v ~ N(0, 1); the log-decay is the
bounded scaled sigmoid g = -5 * sigmoid(x_g) with x_g ~ N(0, 1), per key channel
(Kimi K3 technical-report digest, section 2.1 (1): g_min = -5); the write gate is
beta = sigmoid(x_b) with x_b ~ N(0, 1), one per (token, head); the initial state
S0 ~ N(0, s0_std^2) in fp32 when asked for.  The draws are made in the order q, k,
v, x_g, x_b, S0 from one generator seeded with ``seed``.

``slow_decay=True`` selects the test-only stress mix (x_g ~ N(-10, 1), so g is
about -2e-4, and x_b ~ N(-6, 1), so beta is about 0.0025): with the standard
mix the state forgets within a few tokens, which would let a wrong initial
state or a wrong segment composition pass unnoticed.
"""
from __future__ import annotations

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _normal(shape, gen, device, mean=0.0, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def _unit_rows(x):
    return x / x.norm(dim=-1, keepdim=True)


def make_prefill_inputs(lengths, H, dk, dv, act="bf16", *, seed=0, s0_std=None,
                        device="cpu", slow_decay=False):
    """Packed variable-length prefill inputs.

    Returns a dict: q, k ``[T, H, dk]`` and v ``[T, H, dv]`` in the activation
    dtype; g ``[T, H, dk]`` and beta ``[T, H]`` fp32; S0 ``[N, H, dk, dv]`` fp32 or
    None; cu_seqlens int32 ``[N+1]`` (on ``device``) and ``lengths``.  The same
    draws before their preparation, for the fused-prologue entry point: q_raw,
    k_raw (not normalised) and x_g in the activation dtype, x_beta fp32.
    """
    lengths = [int(x) for x in lengths]
    T = sum(lengths)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = DTYPES[act]
    # each fp32 draw is turned into what is kept before the next one is made, so
    # at most two fp32 copies of one array exist at a time (a 1M-token x 56-head
    # workload stays well inside device memory)
    x = _normal((T, H, dk), gen, device)
    q, q_raw = _unit_rows(x).to(dt), x.to(dt)
    x = _normal((T, H, dk), gen, device)
    k, k_raw = _unit_rows(x).to(dt), x.to(dt)
    del x
    v = _normal((T, H, dv), gen, device).to(dt)
    xg = _normal((T, H, dk), gen, device, mean=-10.0 if slow_decay else 0.0)
    x_g = xg.to(dt).contiguous()
    g = torch.sigmoid(xg).mul_(-5.0)
    del xg
    xb = _normal((T, H), gen, device, mean=-6.0 if slow_decay else 0.0)
    beta = torch.sigmoid(xb)
    S0 = None
    if s0_std is not None:
        S0 = _normal((len(lengths), H, dk, dv), gen, device, std=float(s0_std))
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    cu_seqlens = torch.tensor(cu, dtype=torch.int32, device=device)
    return {"q": q, "k": k, "v": v, "g": g.contiguous(), "beta": beta.contiguous(),
            "S0": S0, "cu_seqlens": cu_seqlens, "lengths": lengths,
            "q_raw": q_raw, "k_raw": k_raw, "x_g": x_g, "x_beta": xb.contiguous()}


def make_backward_adjoints(T, N, H, dk, dv, act="bf16", *, seed=0, device="cpu",
                           final=True):
    """Adjoints for the backward pass: d_out ``[T, H, dv]`` ~ N(0, 1) in the
    activation dtype and, if ``final``, d_S_final ``[N, H, dk, dv]`` ~ N(0, 1) fp32
    (else None), drawn in that order from one generator seeded with ``seed``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    d_out = _normal((T, H, dv), gen, device).to(DTYPES[act])
    d_sf = _normal((N, H, dk, dv), gen, device) if final else None
    return d_out, d_sf


def make_decode_inputs(batch, H, dk, dv, steps, act="bf16", *, seed=0, s0_std=0.02,
                       device="cpu", slow_decay=False):
    """``steps`` successive single-token inputs for ``batch`` sequences.

    Returns a dict: q, k ``[steps, batch, H, dk]``, v ``[steps, batch, H, dv]`` in
    the activation dtype; g ``[steps, batch, H, dk]``, beta ``[steps, batch, H]``
    fp32; S0 ``[batch, H, dk, dv]`` fp32 (N(0, s0_std^2)).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = DTYPES[act]
    q = _unit_rows(_normal((steps, batch, H, dk), gen, device)).to(dt)
    k = _unit_rows(_normal((steps, batch, H, dk), gen, device)).to(dt)
    v = _normal((steps, batch, H, dv), gen, device).to(dt)
    xg = _normal((steps, batch, H, dk), gen, device, mean=-10.0 if slow_decay else 0.0)
    xb = _normal((steps, batch, H), gen, device, mean=-6.0 if slow_decay else 0.0)
    g = (-5.0 * torch.sigmoid(xg)).contiguous()
    beta = torch.sigmoid(xb).contiguous()
    S0 = _normal((batch, H, dk, dv), gen, device, std=float(s0_std))
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "S0": S0}


# The five workloads, by what they are.  Sizes follow the published configs.
WORKLOADS = {
    "kda_fwd_f32_h2_t64_d16": dict(kind="prefill", lengths=[64], H=2, dk=16, dv=16,
                                   act="f32", s0_std=None),
    "kda_prefill_bf16_h8_t4096_d128": dict(kind="prefill", lengths=[4096], H=8, dk=128,
                                           dv=128, act="bf16", s0_std=None),
    "kda_prefill_varlen4_h56_t81920_d128_s0": dict(kind="prefill",
                                                   lengths=[8192, 16384, 24576, 32768],
                                                   H=56, dk=128, dv=128, act="bf16",
                                                   s0_std=0.02),
    "kda_decode_b256_h56_d128_x64": dict(kind="decode", batch=256, H=56, dk=128, dv=128,
                                         steps=64, act="bf16", s0_std=0.02),
    "kda_prefill_kcp64_h56_t1m_d128": dict(kind="prefill", lengths=[1048576], H=56,
                                           dk=128, dv=128, act="bf16", s0_std=None,
                                           num_segments=64),
}
