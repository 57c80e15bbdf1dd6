"""KCP across ranks with the libkda steps on one GPU: W ranks emulated in one
process (each rank's transfer pass, the concatenation an all-gather would give,
the local scan and each rank's segment pass), against the oracle's whole-batch
recurrence.  (A multi-rank run needs one GPU per rank.)"""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_18_gb300 import kcp
from kimi_delta_attention_18_gb300.inputs import make_prefill_inputs
from tests.conftest import rel_err

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.mark.parametrize("act,d,W", [("f32", 32, 2), ("f32", 32, 5), ("bf16", 128, 4)])
def test_kcp_emulated_ranks_on_gpu(act, d, W):
    lengths = [700, 90, 0, 333]
    H = 2
    x = make_prefill_inputs(lengths, H, d, d, act, s0_std=1.0, seed=52, slow_decay=True)
    x = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    args = (x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"])
    pairs = [kcp.local_pairs(*args, W, r) for r in range(W)]
    A_all = torch.stack([p[0] for p in pairs], dim=2)
    B_all = torch.stack([p[1] for p in pairs], dim=2)
    T = x["q"].shape[0]
    out = torch.zeros((T, H, d), dtype=torch.float64)
    finals = []
    for r in range(W):
        o, f = kcp.finish(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["cu_seqlens"],
                          W, r, A_all, B_all)
        m = kcp.segment_token_mask(x["cu_seqlens"], W, r, T)
        out[m] = o.double().cpu()[m]
        finals.append(f)
    torch.cuda.synchronize()
    f64 = lambda t: t.detach().float().cpu().double().numpy()
    o_ref, S_ref = oracle.kda_forward(*(f64(x[n]) for n in ("q", "k", "v", "g", "beta")),
                                      f64(x["S0"]), x["cu_seqlens"].cpu().numpy())
    assert rel_err(out.numpy(), o_ref) <= TOL[act]
    for f in finals:
        assert rel_err(f64(f), S_ref) <= TOL[act]
