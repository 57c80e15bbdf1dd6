"""The allocation-free prefill entry point (for callers that may not call
cudaMalloc, e.g. an engine plugin enqueueing work into memory it was handed up
front) must give what the ordinary one-call prefill gives, and what the fp64
oracle gives.

Called through the C ABI twice in a row, on different inputs, so that whatever
the first call leaves in the library's shared scratch cannot leak into the
second.  Kept in its own file, named to be collected last.
"""
import ctypes

import pytest
import torch

import oracle
import kimi_delta_attention_18_gb300 as kda
from kimi_delta_attention_18_gb300.inputs import make_prefill_inputs
from tests.conftest import rel_err

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 * 1024 * 1024
TOL = 2e-2  # BF16 activations, as in the other parity tests


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(x, nseg, out, SF, status):
    desc = kda.prefill_desc(x["q"], x["v"], x["cu_seqlens"], nseg)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return kda.lib().kda_prefill_chunked_noalloc(
        ctypes.byref(desc), _ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["g"]),
        _ptr(x["beta"]), _ptr(x["S0"]), _ptr(x["cu_seqlens"]), _ptr(out), _ptr(SF),
        _ptr(status), stream)


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    cases = [([4096], 8, 32, 0),                 # the H8 T4096 workload, 32 segments
             ([1500, 700, 333], 4, 8, 1)]        # varlen with an initial state, 8 segments
    for lengths, H, nseg, seed in cases:
        x = make_prefill_inputs(lengths, H, 128, 128, "bf16", seed=seed,
                                s0_std=0.5 if seed else None, device="cuda", slow_decay=bool(seed))
        desc = kda.prefill_desc(x["q"], x["v"], x["cu_seqlens"], nseg)
        assert 0 < kda.prefill_workspace_size(desc) <= SCRATCH_BYTES
        ref_out, ref_SF = kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"],
                                              x["cu_seqlens"], num_segments=nseg)
        out = torch.full_like(ref_out, float("nan"))
        SF = torch.full_like(ref_SF, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(x, nseg, out, SF, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rel_err(out.float().cpu().numpy(), ref_out.float().cpu().numpy()) <= TOL
        assert rel_err(SF.cpu().numpy(), ref_SF.cpu().numpy()) <= TOL
        # and directly against the oracle on the same inputs
        f = lambda t: None if t is None else t.detach().float().cpu().double().numpy()
        o_ref, S_ref = oracle.kda_forward(*(f(x[n]) for n in ("q", "k", "v", "g", "beta")),
                                          f(x["S0"]), x["cu_seqlens"].cpu().numpy())
        assert rel_err(out.float().cpu().numpy(), o_ref) <= TOL
        assert rel_err(SF.cpu().numpy(), S_ref) <= TOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    x = make_prefill_inputs([64], 1, 128, 128, "bf16", device="cuda")
    # 600 segments x (A, B, start state) of 64 KB each need 112.5 MiB > 64 MiB
    desc = kda.PrefillDesc(1, 64, 1, 128, 128, 1, 16, 600)
    assert kda.prefill_workspace_size(desc) > SCRATCH_BYTES
    rc = kda.lib().kda_prefill_chunked_noalloc(
        ctypes.byref(desc), _ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["g"]),
        _ptr(x["beta"]), None, _ptr(x["cu_seqlens"]), _ptr(x["v"]), None, None, None)
    assert rc == 3  # KDA_ERR_WORKSPACE, nothing launched
