"""GPU parity of the fused gate prologue and of the sparse state checkpoints at the
long-context size and launch configuration the bench times: 1,048,576 tokens x 56
heads, d = 128, BF16, 64 segments (the two-chain transfer pass with a lead segment
run from S0, the scan and the combine), with S0 ~ N(0, 1).  Sampled heads against
the oracle; checkpoints on both sides of the lead segment's end, the last one being
the final state."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_18_gb300 as kda
from kimi_delta_attention_18_gb300.inputs import WORKLOADS, make_prefill_inputs
from tests.conftest import rel_err

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not kda.lib().kda_build_info().decode().endswith("tc:1"),
                       reason="needs the tensor-core prefill (the CUDA-core path is too slow "
                              "at 1M x 56)"),
]

W = WORKLOADS["kda_prefill_kcp64_h56_t1m_d128"]


def _np(t):
    return None if t is None else t.detach().float().cpu().double().numpy()


def _inputs(seed):
    x = make_prefill_inputs(W["lengths"], W["H"], W["dk"], W["dv"], W["act"], s0_std=1.0,
                            seed=seed, device="cuda")
    return x


def _heads(x, names, heads):
    sel = torch.tensor(heads, device="cuda")
    return [_np(x[n][:, sel]) for n in names]


def test_gated_headline_size_sampled_heads():
    x = _inputs(41)
    out, SF = kda.prefill_chunked_gated(x["q_raw"], x["k_raw"], x["v"], x["x_g"], x["x_beta"],
                                        x["S0"], x["cu_seqlens"],
                                        num_segments=W["num_segments"])
    torch.cuda.synchronize()
    assert torch.isfinite(SF).all()
    heads = [5, 38]
    q_raw, k_raw, v, x_g, x_beta = _heads(x, ("q_raw", "k_raw", "v", "x_g", "x_beta"), heads)
    S0 = _heads(x, ("S0",), heads)[0]
    qn, kn, g, beta = oracle.gate_prologue(q_raw, k_raw, x_g, x_beta)
    o_ref, S_ref = oracle.kda_forward(qn, kn, v, g, beta, S0, x["cu_seqlens"].cpu().numpy())
    sel = torch.tensor(heads, device="cuda")
    assert rel_err(_np(SF[:, sel]), S_ref) <= 2e-2
    step = 3001  # tokens in the lead segment, in the transfer segments and at their joins
    o = _np(out[::step][:, sel])
    assert np.isfinite(o).all()
    assert rel_err(o, o_ref[::step]) <= 2e-2


def test_checkpoints_headline_size_sampled_head():
    x = _inputs(42)
    interval = 4096
    out, SF, ck = kda.prefill_chunked_ckpt(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"],
                                           x["cu_seqlens"], ckpt_interval=interval,
                                           num_segments=W["num_segments"])
    torch.cuda.synchronize()
    T = W["lengths"][0]
    assert ck.shape[0] == T // interval == kda.num_checkpoints(x["cu_seqlens"], interval)
    h = 23
    q, k, v, g, b = _heads(x, ("q", "k", "v", "g", "beta"), [h])
    S = _heads(x, ("S0",), [h])[0]
    # the lead segment (segment 0, run from S0) ends near token 0.48 T with 56 chains on
    # 152 SMs: checkpoints 1 and 100 fall inside it, 130 and 200 in transfer segments,
    # 256 is the last token (the final state)
    done = 0
    for kk in (1, 100, 130, 200, 256):
        p = kk * interval
        sl = slice(done, p)
        _, S = oracle.kda_forward(q[sl], k[sl], v[sl], g[sl], b[sl], S,
                                  np.array([0, p - done], dtype=np.int32))
        done = p
        assert rel_err(_np(ck[kk - 1, h]), S[0, 0]) <= 2e-2, kk
    assert rel_err(_np(SF[0, h]), S[0, 0]) <= 2e-2
    # the last checkpoint (through the fix-up) and the final state (through the scan)
    assert rel_err(_np(ck[-1]), _np(SF[0])) <= 2e-2
