"""GPU parity of the sparse state checkpoints (kda_prefill_chunked_ckpt): every
checkpoint against the oracle's final state of that sequence truncated after the
checkpoint's token count, on one pass and on the split path (segment
boundaries inside and between checkpoints), with a material initial state
(slow forgetting) so that a missing start-state term cannot pass."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_18_gb300 as kda
from kimi_delta_attention_18_gb300.inputs import make_prefill_inputs
from tests.conftest import rel_err

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def _np(t):
    return t.detach().float().cpu().double().numpy()


@pytest.mark.parametrize("act,d,interval,nseg", [
    ("bf16", 128, 256, 1), ("bf16", 128, 256, 4), ("bf16", 128, 112, 8), ("bf16", 128, 64, 0),
    # 8 chains x 20 segments fill the SMs: two-chain transfer pass with a lead segment
    # (the first blocks of the 700-token sequence, run from S0, hold a checkpoint)
    ("bf16", 128, 32, 20),
    ("f32", 32, 64, 1), ("f32", 32, 48, 3),
])
def test_checkpoints_match_oracle_prefix_states(act, d, interval, nseg):
    lengths = [700, 333, 45, 256]
    H = 2
    x = make_prefill_inputs(lengths, H, d, d, act, s0_std=1.0, seed=21, slow_decay=True)
    x = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    out, SF, ck = kda.prefill_chunked_ckpt(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"],
                                           x["cu_seqlens"], ckpt_interval=interval,
                                           num_segments=nseg)
    out0, SF0 = kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"],
                                    x["cu_seqlens"], num_segments=nseg)
    torch.cuda.synchronize()
    # the checkpoints change nothing else
    assert torch.equal(out, out0) and torch.equal(SF, SF0)
    cu = x["cu_seqlens"].cpu().tolist()
    q, k, v, g, b, S0 = (_np(x[n]) for n in ("q", "k", "v", "g", "beta", "S0"))
    ck = _np(ck)
    slot = 0
    for n, L in enumerate(lengths):
        for kk in range(L // interval):
            p = (kk + 1) * interval
            sl = slice(cu[n], cu[n] + p)
            _, S_ref = oracle.kda_forward(q[sl], k[sl], v[sl], g[sl], b[sl], S0[n:n + 1],
                                          np.array([0, p], dtype=np.int32))
            assert rel_err(ck[slot], S_ref[0]) <= TOL[act], (n, kk)
            if p == L:  # a checkpoint at the sequence's last token is its final state
                assert rel_err(ck[slot], _np(SF[n])) <= TOL[act]
            slot += 1
    assert ck.shape[0] == slot == kda.num_checkpoints(x["cu_seqlens"], interval)


def test_no_checkpoint_due():
    x = make_prefill_inputs([40, 17], 2, 128, 128, "bf16", seed=22)
    x = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    out, SF, ck = kda.prefill_chunked_ckpt(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                           x["cu_seqlens"], ckpt_interval=64)
    torch.cuda.synchronize()
    assert ck.shape[0] == 0 and torch.isfinite(SF).all()
