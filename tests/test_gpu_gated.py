"""GPU parity of the fused gate prologue (kda_prefill_chunked_gated): the prefill
from raw q, k, the gate pre-activations x_g (BF16) and x_beta against the fp64
oracle run on the oracle's own prologue of the same values, on one pass and on
the split path; and against kda_prefill_chunked on inputs prepared outside."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_18_gb300 as kda
from kimi_delta_attention_18_gb300.inputs import make_prefill_inputs
from tests.conftest import rel_err

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().double().numpy()


@pytest.mark.parametrize("nseg,slow", [(1, False), (1, True), (4, True), (8, False), (20, True)])
def test_gated_prefill_matches_oracle(nseg, slow):
    lengths = [700, 333, 45, 256]
    H = 2
    x = make_prefill_inputs(lengths, H, 128, 128, "bf16", s0_std=1.0, seed=31, slow_decay=slow)
    x = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    out, SF = kda.prefill_chunked_gated(x["q_raw"], x["k_raw"], x["v"], x["x_g"], x["x_beta"],
                                        x["S0"], x["cu_seqlens"], num_segments=nseg)
    torch.cuda.synchronize()
    qn, kn, g, beta = oracle.gate_prologue(_np(x["q_raw"]), _np(x["k_raw"]), _np(x["x_g"]),
                                           _np(x["x_beta"]))
    o_ref, S_ref = oracle.kda_forward(qn, kn, _np(x["v"]), g, beta, _np(x["S0"]),
                                      x["cu_seqlens"].cpu().numpy())
    assert rel_err(_np(out), o_ref) <= 2e-2
    assert rel_err(_np(SF), S_ref) <= 2e-2
    # the same as the plain entry point on inputs prepared in fp32 outside
    qp = (x["q_raw"].float() / x["q_raw"].float().norm(dim=-1, keepdim=True)).bfloat16()
    kp = (x["k_raw"].float() / x["k_raw"].float().norm(dim=-1, keepdim=True)).bfloat16()
    gp = (-5.0 * torch.sigmoid(x["x_g"].float())).contiguous()
    bp = torch.sigmoid(x["x_beta"]).contiguous()
    out2, SF2 = kda.prefill_chunked(qp, kp, x["v"], gp, bp, x["S0"], x["cu_seqlens"],
                                    num_segments=nseg)
    torch.cuda.synchronize()
    assert rel_err(_np(out), _np(out2)) <= 2e-2 and rel_err(_np(SF), _np(SF2)) <= 2e-2


def test_gated_zero_rows_stay_finite():
    x = make_prefill_inputs([64], 1, 128, 128, "bf16", seed=32)
    x = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    q = x["q_raw"].clone()
    k = x["k_raw"].clone()
    q[5].zero_()
    k[9].zero_()
    out, SF = kda.prefill_chunked_gated(q, k, x["v"], x["x_g"], x["x_beta"], None,
                                        x["cu_seqlens"], num_segments=1)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(SF).all()
    qn, kn, g, beta = oracle.gate_prologue(_np(q), _np(k), _np(x["x_g"]), _np(x["x_beta"]))
    o_ref, S_ref = oracle.kda_forward(qn, kn, _np(x["v"]), g, beta, None,
                                      x["cu_seqlens"].cpu().numpy())
    assert rel_err(_np(out), o_ref) <= 2e-2 and rel_err(_np(SF), S_ref) <= 2e-2


def test_gated_lead_path_with_zero_rows():
    # 8 chains x 20 segments: the two-chain transfer pass with a lead segment, whose
    # CTAs take the norms and the gate from their helper warps; zero rows inside
    # and outside the lead, and a ragged tail
    x = make_prefill_inputs([1000, 37], 4, 128, 128, "bf16", s0_std=1.0, seed=33, slow_decay=True)
    x = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    q = x["q_raw"].clone()
    k = x["k_raw"].clone()
    q[5].zero_()
    k[9].zero_()
    k[700, 2].zero_()
    out, SF = kda.prefill_chunked_gated(q, k, x["v"], x["x_g"], x["x_beta"], x["S0"],
                                        x["cu_seqlens"], num_segments=20)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(SF).all()
    qn, kn, g, beta = oracle.gate_prologue(_np(q), _np(k), _np(x["x_g"]), _np(x["x_beta"]))
    o_ref, S_ref = oracle.kda_forward(qn, kn, _np(x["v"]), g, beta, _np(x["S0"]),
                                      x["cu_seqlens"].cpu().numpy())
    assert rel_err(_np(out), o_ref) <= 2e-2 and rel_err(_np(SF), S_ref) <= 2e-2
