"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same
seeded inputs (the oracle gets the activation-dtype values upcast to fp64).

Bound (relative to the tensor's largest magnitude, per tensor, for outputs and
final states alike): 1e-4 with fp32 activations, 2e-2 with BF16 activations
(fp32 gates, accumulation and state).
"""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_18_gb300 as kda
from kimi_delta_attention_18_gb300.inputs import WORKLOADS, make_decode_inputs, make_prefill_inputs
from tests.conftest import rel_err

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def _np(t):
    return None if t is None else t.detach().float().cpu().double().numpy()


def _oracle_prefill(x, heads=None, S0=None):
    """Oracle on the host copy of x, optionally restricted to some heads (sliced on
    the device first, so a full-size workload never crosses to the host)."""
    sel = slice(None) if heads is None else torch.tensor(heads, device=x["q"].device)
    q, k, v, g, b = (_np(x[n][:, sel]) for n in ("q", "k", "v", "g", "beta"))
    if S0 is None and x["S0"] is not None:
        S0 = _np(x["S0"][:, sel])
    return oracle.kda_forward(q, k, v, g, b, S0, x["cu_seqlens"].cpu().numpy())


def _gpu_inputs(lengths, H, dk, dv, act, **kw):
    x = make_prefill_inputs(lengths, H, dk, dv, act, **kw)
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


def _run(x, num_segments=0, S0="x"):
    S0 = x["S0"] if S0 == "x" else S0
    out, SF = kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], S0,
                                  x["cu_seqlens"], num_segments=num_segments)
    torch.cuda.synchronize()
    return out, SF


def test_config0_fp32_matches_oracle():
    w = WORKLOADS["kda_fwd_f32_h2_t64_d16"]
    x = _gpu_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"])
    out, SF = _run(x)
    o_ref, S_ref = _oracle_prefill(x)
    assert rel_err(_np(out), o_ref) <= 1e-4
    assert rel_err(_np(SF), S_ref) <= 1e-4


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("slow", [False, True])
def test_fp32_varlen_ragged_with_initial_state(d, slow):
    lengths = [37, 0, 16, 5, 50, 1, 17]
    x = _gpu_inputs(lengths, 3, d, d, "f32", s0_std=0.02 if not slow else 1.0, seed=d,
                    slow_decay=slow)
    out, SF = _run(x)
    o_ref, S_ref = _oracle_prefill(x)
    assert rel_err(_np(out), o_ref) <= 1e-4
    assert rel_err(_np(SF), S_ref) <= 1e-4


def test_fp32_unequal_dk_dv_and_split():
    x = _gpu_inputs([100, 61], 2, 24, 40, "f32", s0_std=0.5, seed=3, slow_decay=True)
    o_ref, S_ref = _oracle_prefill(x)
    for nseg in (1, 3, 7):
        out, SF = _run(x, nseg)
        assert rel_err(_np(out), o_ref) <= 1e-4, nseg
        assert rel_err(_np(SF), S_ref) <= 1e-4, nseg


def test_config1_bf16_full_matches_oracle():
    w = WORKLOADS["kda_prefill_bf16_h8_t4096_d128"]
    x = _gpu_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"])
    o_ref, S_ref = _oracle_prefill(x)
    for nseg in (0, 1):  # the chosen split (as timed) and the single pass
        out, SF = _run(x, nseg)
        assert rel_err(_np(out), o_ref) <= 2e-2, nseg
        assert rel_err(_np(SF), S_ref) <= 2e-2, nseg


@pytest.mark.parametrize("nseg", [1, 8, 32])
def test_bf16_slow_decay_initial_state_and_split(nseg):
    """Slow forgetting keeps S0 and every segment's transfer matrix material, so a
    wrong start state or a wrong composition cannot pass."""
    x = _gpu_inputs([1024, 700, 333], 4, 128, 128, "bf16", s0_std=1.0, seed=11, slow_decay=True)
    o_ref, S_ref = _oracle_prefill(x)
    out, SF = _run(x, nseg)
    assert rel_err(_np(out), o_ref) <= 2e-2
    assert rel_err(_np(SF), S_ref) <= 2e-2
    # the initial state matters here: dropping it must break parity
    out0, SF0 = _run(x, nseg, S0=None)
    assert rel_err(_np(SF0), S_ref) > 0.1


@pytest.mark.parametrize("nseg", [0, 1])
def test_config1_shape_slow_decay_with_initial_state(nseg):
    """The short-prefill shape (H = 8, T = 4096) with slow forgetting and S0 ~
    N(0, 1): S0 and every segment's transfer matrix stay material over the whole
    sequence, so the chosen split (nseg = 0) and the single pass are both held to
    the oracle on every head, and dropping S0 must break parity."""
    x = _gpu_inputs([4096], 8, 128, 128, "bf16", s0_std=1.0, seed=21, slow_decay=True,
                    device="cuda")
    o_ref, S_ref = _oracle_prefill(x)
    out, SF = _run(x, nseg)
    assert rel_err(_np(out), o_ref) <= 2e-2
    assert rel_err(_np(SF), S_ref) <= 2e-2
    _, SF0 = _run(x, nseg, S0=None)
    assert rel_err(_np(SF0), S_ref) > 0.1


def test_config4_shape_slow_decay_64_segments_sampled_heads():
    """The long-context shape (H = 56, 64 segments) at a reduced length (64 x 128
    tokens) with slow forgetting and S0 ~ N(0, 1): every segment's start state is
    the composition of all the segments before it, so a wrong transfer matrix or a
    wrong scan step shows.  Sampled heads against the oracle; dropping S0 must
    break parity.  (The stress mix has E[g] of about -3.7e-4 per token, so S0
    still carries about e^-3 of its weight after 8192 tokens, far above the written
    part's share; at 16K tokens it would be e^-6.)"""
    T, H, nseg = 64 * 128, 56, 64
    x = _gpu_inputs([T], H, 128, 128, "bf16", s0_std=1.0, seed=22, slow_decay=True,
                    device="cuda")
    out, SF = _run(x, nseg)
    heads = [3, 40]
    o_ref, S_ref = _oracle_prefill(x, heads=heads)
    assert rel_err(_np(out[:, heads]), o_ref) <= 2e-2
    assert rel_err(_np(SF[:, heads]), S_ref) <= 2e-2
    assert torch.isfinite(out.float()).all() and torch.isfinite(SF).all()
    _, SF0 = _run(x, nseg, S0=None)
    assert rel_err(_np(SF0[:, heads]), S_ref) > 0.1


@pytest.mark.parametrize("gated", [False, True])
def test_two_chain_transfer_pass_ragged(gated):
    """Enough segments (N x H x S = 3 x 16 x 4 = 192, at least one per SM) that the
    transfer pass runs a segment's identity-start and zero-start chains in one CTA
    from one prep; ragged lengths with partial last blocks, slow forgetting and
    S0 ~ N(0, 1), plain and from the gate pre-activations, against the oracle."""
    lengths = [300, 45, 130]
    H, nseg = 16, 4
    x = _gpu_inputs(lengths, H, 128, 128, "bf16", s0_std=1.0, seed=17, slow_decay=True,
                    device="cuda")
    assert len(lengths) * H * nseg >= torch.cuda.get_device_properties(0).multi_processor_count
    if gated:
        out, SF = kda.prefill_chunked_gated(x["q_raw"], x["k_raw"], x["v"], x["x_g"],
                                            x["x_beta"], x["S0"], x["cu_seqlens"],
                                            num_segments=nseg)
        torch.cuda.synchronize()
        qn, kn, g, beta = oracle.gate_prologue(_np(x["q_raw"]), _np(x["k_raw"]), _np(x["x_g"]),
                                               _np(x["x_beta"]))
        o_ref, S_ref = oracle.kda_forward(qn, kn, _np(x["v"]), g, beta, _np(x["S0"]),
                                          x["cu_seqlens"].cpu().numpy())
    else:
        out, SF = _run(x, nseg)
        o_ref, S_ref = _oracle_prefill(x)
    assert torch.isfinite(out.float()).all() and torch.isfinite(SF).all()
    assert rel_err(_np(out), o_ref) <= 2e-2
    assert rel_err(_np(SF), S_ref) <= 2e-2
    if not gated:  # the stage entry point in the same regime: A, B against the oracle
        A, B = kda.state_transfer(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], nseg)
        torch.cuda.synchronize()
        A_ref, B_ref = oracle.kda_state_transfer(_np(x["k"]), _np(x["v"]), _np(x["g"]),
                                                 _np(x["beta"]), x["cu_seqlens"].cpu().numpy(),
                                                 nseg)
        assert rel_err(_np(A), A_ref) <= 2e-2 and rel_err(_np(B), B_ref) <= 2e-2


def test_lead_segment_with_empty_and_short_sequences():
    """The lead regime (120 chains, fewer than the SMs; 4 segments, so at least one
    unit per SM): the first segment of every chain is longer and runs from S0 beside
    the transfer pass.  Empty sequences (every segment empty: the final state is S0
    itself), a sequence shorter than one block and ragged ones, with slow forgetting
    and S0 ~ N(0, 1), against the oracle; dropping S0 must break parity."""
    lengths = [0, 200, 0, 7, 61]
    H, nseg = 24, 4
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert len(lengths) * H < sms <= len(lengths) * H * nseg
    x = _gpu_inputs(lengths, H, 128, 128, "bf16", s0_std=1.0, seed=23, slow_decay=True,
                    device="cuda")
    out, SF = _run(x, nseg)
    o_ref, S_ref = _oracle_prefill(x)
    assert torch.isfinite(out.float()).all() and torch.isfinite(SF).all()
    assert rel_err(_np(out), o_ref) <= 2e-2
    assert rel_err(_np(SF), S_ref) <= 2e-2
    # an empty sequence hands its initial state through unchanged, up to the scan's
    # hi/lo BF16 split of each state (about 2^-16 of it per segment step)
    for n in (0, 2):
        assert rel_err(_np(SF[n]), _np(x["S0"][n])) <= 1e-4
    _, SF0 = _run(x, nseg, S0=None)
    assert rel_err(_np(SF0), S_ref) > 0.1


def test_config2_varlen_full_size_sampled_heads():
    w = WORKLOADS["kda_prefill_varlen4_h56_t81920_d128_s0"]
    x = _gpu_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"], s0_std=w["s0_std"],
                    device="cuda")
    out, SF = _run(x)
    heads = [0, 37]
    o_ref, S_ref = _oracle_prefill(x, heads=heads)
    assert rel_err(_np(out[:, heads]), o_ref) <= 2e-2
    assert rel_err(_np(SF[:, heads]), S_ref) <= 2e-2
    assert torch.isfinite(out.float()).all() and torch.isfinite(SF).all()


def test_config3_decode_64_steps_sampled_sequences():
    w = WORKLOADS["kda_decode_b256_h56_d128_x64"]
    x = make_decode_inputs(w["batch"], w["H"], w["dk"], w["dv"], w["steps"], w["act"],
                           s0_std=w["s0_std"], device="cuda")
    S = x["S0"].clone()
    outs = []
    for t in range(w["steps"]):
        outs.append(kda.decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S))
    torch.cuda.synchronize()
    seqs = list(range(0, 256, 37))
    Sr = _np(x["S0"])[seqs]
    for t in range(w["steps"]):
        o_ref, Sr = oracle.kda_decode_step(*(_np(x[n][t])[seqs] for n in ("q", "k", "v", "g", "beta")),
                                           Sr)
        assert rel_err(_np(outs[t])[seqs], o_ref) <= 2e-2, t
    assert rel_err(_np(S)[seqs], Sr) <= 1e-4


def test_decode_continues_prefill():
    """Prefill of T tokens followed by n decode steps equals prefill of T + n tokens."""
    T, n, H = 200, 5, 3
    x = _gpu_inputs([T + n], H, 128, 128, "bf16", s0_std=1.0, seed=5, slow_decay=True)
    full_out, full_S = _run(x)
    part = {k_: (v_[:T] if k_ in ("q", "k", "v", "g", "beta") else v_) for k_, v_ in x.items()}
    part["cu_seqlens"] = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    _, S = _run(part)
    for t in range(T, T + n):
        o = kda.decode_step(x["q"][t:t + 1], x["k"][t:t + 1], x["v"][t:t + 1], x["g"][t:t + 1],
                            x["beta"][t:t + 1], S)
        assert rel_err(_np(o[0]), _np(full_out[t])) <= 2e-2
    torch.cuda.synchronize()
    assert rel_err(_np(S), _np(full_S)) <= 2e-2


def test_resume_from_saved_state():
    """Prefix caching: prefill(0:a), then prefill(a:T) from the saved state."""
    T, a, H = 900, 368, 2
    x = _gpu_inputs([T], H, 128, 128, "bf16", s0_std=1.0, seed=6, slow_decay=True)
    o_ref, S_ref = _oracle_prefill(x)
    first = {k_: (v_[:a] if k_ in ("q", "k", "v", "g", "beta") else v_) for k_, v_ in x.items()}
    first["cu_seqlens"] = torch.tensor([0, a], dtype=torch.int32, device="cuda")
    second = {k_: (v_[a:].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
              for k_, v_ in x.items()}
    second["cu_seqlens"] = torch.tensor([0, T - a], dtype=torch.int32, device="cuda")
    o1, S1 = _run(first)
    o2, S2 = _run(second, S0=S1)
    assert rel_err(np.concatenate([_np(o1), _np(o2)]), o_ref) <= 2e-2
    assert rel_err(_np(S2), S_ref) <= 2e-2


def test_packing_equals_separate_calls():
    lengths = [130, 16, 0, 77]
    x = _gpu_inputs(lengths, 2, 128, 128, "bf16", s0_std=0.5, seed=8, slow_decay=True)
    out, SF = _run(x)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    for n, L in enumerate(lengths):
        xs = {k_: (v_[cu[n]:cu[n + 1]].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
              for k_, v_ in x.items()}
        xs["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32, device="cuda")
        o, S = _run(xs, S0=x["S0"][n:n + 1].contiguous())
        if L:
            assert rel_err(_np(o), _np(out[cu[n]:cu[n + 1]])) <= 1e-6
        assert rel_err(_np(S), _np(SF[n:n + 1])) <= 1e-6


@pytest.mark.parametrize("act,d", [("f32", 32), ("bf16", 128)])
def test_transfer_and_compose_entry_points(act, d):
    lengths = [300, 45]
    nseg = 5
    x = _gpu_inputs(lengths, 2, d, d, act, s0_std=1.0, seed=9, slow_decay=True)
    A, B = kda.state_transfer(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], nseg)
    torch.cuda.synchronize()
    cu = x["cu_seqlens"].cpu().numpy()
    A_ref, B_ref = oracle.kda_state_transfer(_np(x["k"]), _np(x["v"]), _np(x["g"]),
                                             _np(x["beta"]), cu, nseg)
    tol = TOL[act]
    assert rel_err(_np(A), A_ref) <= tol and rel_err(_np(B), B_ref) <= tol
    starts, SF = kda.state_compose(A.reshape(4, nseg, d, d), B.reshape(4, nseg, d, d),
                                   x["S0"].reshape(4, d, d))
    st_ref, SF_ref = oracle.kda_state_compose(_np(A).reshape(4, nseg, d, d),
                                              _np(B).reshape(4, nseg, d, d),
                                              _np(x["S0"]).reshape(4, d, d))
    torch.cuda.synchronize()
    assert rel_err(_np(starts), st_ref) <= 1e-5 and rel_err(_np(SF), SF_ref) <= 1e-5
    out, SF2 = kda.prefill_segments(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                    starts.reshape(2, 2, nseg, d, d), x["cu_seqlens"], nseg)
    o_ref, S_ref = _oracle_prefill(x)
    torch.cuda.synchronize()
    assert rel_err(_np(out), o_ref) <= tol and rel_err(_np(SF2), S_ref) <= tol


def test_edge_cases_empty_tiny_and_in_place():
    for lengths in ([0], [0, 0, 0], [1], [15], [16], [17], [0, 1, 0, 33]):
        x = _gpu_inputs(lengths, 2, 128, 128, "bf16", s0_std=1.0, seed=len(lengths))
        S0 = x["S0"].clone()
        out, SF = kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"],
                                      x["cu_seqlens"], S_final=x["S0"])  # in place
        torch.cuda.synchronize()
        o_ref, S_ref = _oracle_prefill(x, S0=_np(S0))
        if sum(lengths):
            assert rel_err(_np(out), o_ref) <= 2e-2
        assert rel_err(_np(SF), S_ref) <= 2e-2
    # N = 0: nothing to do
    x = _gpu_inputs([5], 1, 16, 16, "f32")
    kda.prefill_chunked(x["q"][:0], x["k"][:0], x["v"][:0], x["g"][:0], x["beta"][:0], None,
                        torch.zeros(1, dtype=torch.int32, device="cuda"))


def test_malformed_cu_seqlens_reported_on_device():
    x = _gpu_inputs([40, 24], 2, 16, 16, "f32")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 50, 40], dtype=torch.int32, device="cuda")  # decreasing
    out = torch.full_like(x["v"], 7.0)
    kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], None, bad, out=out,
                        dev_status=status, num_segments=1)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    bad2 = torch.tensor([0, 30, 99], dtype=torch.int32, device="cuda")  # past T_tot
    status.zero_()
    kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], None, bad2, out=out,
                        dev_status=status, num_segments=4)
    torch.cuda.synchronize()
    assert int(status.item()) == 1


@pytest.mark.skipif(not kda.lib().kda_build_info().decode().endswith("tc:1"),
                    reason="needs the tensor-core prefill (the CUDA-core path is too slow at 1M x 56)")
def test_config4_kcp_matches_sequential_and_oracle_head():
    """1M tokens x 56 heads, 64 segments joined by the transfer-matrix scan: every
    head against the single pass on the GPU; one head against the oracle."""
    w = WORKLOADS["kda_prefill_kcp64_h56_t1m_d128"]
    x = _gpu_inputs(w["lengths"], w["H"], w["dk"], w["dv"], w["act"], device="cuda")
    out_k, S_k = _run(x, w["num_segments"])
    out_s, S_s = _run(x, 1)
    assert rel_err(_np(S_k), _np(S_s)) <= 2e-2
    step = 4099
    assert rel_err(_np(out_k[::step]), _np(out_s[::step])) <= 2e-2
    h = 17
    o_ref, S_ref = _oracle_prefill(x, heads=[h])
    assert rel_err(_np(S_k[:, [h]]), S_ref) <= 2e-2
    assert rel_err(_np(out_k[::step, [h]]), o_ref[::step]) <= 2e-2


@pytest.mark.parametrize("nseg", [1, 4, 8])
def test_partial_last_blocks_on_fresh_stages(nseg):
    """Segments of one to three blocks whose last block is partial: the rows past
    the end are weighted by zero on the tensor cores, so they must never carry
    stale shared-memory contents (0 * NaN = NaN).  Outputs start as NaN so a row
    left unwritten cannot hide behind a reused buffer."""
    lengths = [333, 45, 29, 7, 100]
    x = _gpu_inputs(lengths, 4, 128, 128, "bf16", s0_std=0.5, seed=13, slow_decay=True)
    o_ref, S_ref = _oracle_prefill(x)
    for _ in range(2):
        out = torch.full_like(x["v"], float("nan"))
        SF = torch.full((len(lengths), 4, 128, 128), float("nan"), device="cuda")
        kda.prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["cu_seqlens"],
                            num_segments=nseg, out=out, S_final=SF)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all() and torch.isfinite(SF).all()
        assert rel_err(_np(out), o_ref) <= 2e-2
        assert rel_err(_np(SF), S_ref) <= 2e-2


@pytest.mark.parametrize("act,d,first", [("f32", 32, 0), ("bf16", 128, 0), ("bf16", 128, 1)])
def test_split_stages_with_output_correction(act, d, first):
    """The split's three stages through their entry points: transfer pass with
    outputs (zero-start outputs and A_t^T q_t), scan, combine; against the
    oracle.  first = 1 runs from S0 = 0, so the first segment needs no correction."""
    lengths = [300, 45, 130]
    nseg = 5
    x = _gpu_inputs(lengths, 2, d, d, act, s0_std=None if first else 1.0, seed=15,
                    slow_decay=True)
    N, H = len(lengths), 2
    A, B, out, aux = kda.state_transfer(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], nseg,
                                        q=x["q"])
    S0 = None if x["S0"] is None else x["S0"].reshape(N * H, d, d)
    # BF16 at d = 128: the scan also writes the start states' BF16 operand images and
    # the combine reads only those (its tcgen05 path); otherwise the fp32 states
    imgs = (torch.empty((N * H, nseg, d * d), dtype=torch.bfloat16, device="cuda")
            if act == "bf16" and d == 128 else None)
    starts, SF = kda.state_compose(A.reshape(N * H, nseg, d, d), B.reshape(N * H, nseg, d, d), S0,
                                   start_images=imgs)
    if imgs is None:
        kda.prefill_combine(out, aux, starts.reshape(N, H, nseg, d, d), x["cu_seqlens"],
                            first_segment=first)
    else:
        out2 = out.clone()
        kda.prefill_combine(out, aux, None, x["cu_seqlens"], first_segment=first,
                            start_images=imgs, num_segments=nseg)
        kda.prefill_combine(out2, aux, starts.reshape(N, H, nseg, d, d), x["cu_seqlens"],
                            first_segment=first)
    torch.cuda.synchronize()
    o_ref, S_ref = _oracle_prefill(x)
    tol = TOL[act]
    assert rel_err(_np(out), o_ref) <= tol
    assert rel_err(_np(SF).reshape(N, H, d, d), S_ref) <= tol
    if imgs is not None:  # the mma.sync path from the fp32 states agrees too
        assert rel_err(_np(out2), o_ref) <= tol


def test_bounded_wait_gives_up_and_reports():
    """A device-side wait that nothing completes gives up after its limit, writes
    KDA_ERR_TIMEOUT (5) to dev_status and leaves the context usable: the next
    prefill runs and matches the oracle."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda._native.selftest_wait_timeout(2000, st)  # ~2 ms
    torch.cuda.synchronize()
    assert int(st.item()) == 5
    x = _gpu_inputs([100, 37], 2, 128, 128, "bf16", seed=41)
    o_ref, S_ref = _oracle_prefill(x)
    out, SF = _run(x, 1)
    assert rel_err(_np(out), o_ref) <= 2e-2 and rel_err(_np(SF), S_ref) <= 2e-2
