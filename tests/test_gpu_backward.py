"""GPU parity of the backward pass (kda_prefill_backward) against the oracle's
fp64 autograd of the token recurrence: every gradient element by element on
ragged multi-sequence batches (several 16-token blocks and a ragged tail per
sequence, a ragged last column block, empty sequences), with a material initial
state and final-state adjoint; at the bench size, two sampled heads against the
oracle and linearity in the adjoints over the whole output."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_18_gb300 as kda
from kimi_delta_attention_18_gb300.inputs import make_backward_adjoints, make_prefill_inputs
from tests.conftest import rel_err

pytestmark = pytest.mark.gpu

# The token-level path (fp32 activations, and BF16 at other widths) computes in
# fp32: the oracle sees the same (BF16-exact) inputs, so the fp32 bound applies.
# BF16 at dk = dv = 128 takes the chunked tensor-core path (BF16 operands, fp32
# accumulation and state), held to the BF16 bound of the forward.
TOL = 1e-4
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def _tol(act, dk, dv):
    return 2e-2 if act == "bf16" and dk == 128 and dv == 128 else TOL


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _run(x, d_out, d_sf, **kw):
    x = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    got = kda.prefill_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"],
                               x["cu_seqlens"], d_out.cuda(),
                               None if d_sf is None else d_sf.cuda(), **kw)
    torch.cuda.synchronize()
    return got


def _oracle(x, d_out, d_sf, heads=None):
    sel = (lambda a: a) if heads is None else (lambda a: a[:, heads])
    q, k, v, g, b = (sel(_np(x[n])) for n in ("q", "k", "v", "g", "beta"))
    N = len(x["lengths"])
    S0 = _np(x["S0"]) if x["S0"] is not None else np.zeros(
        (N, x["q"].shape[1], x["q"].shape[2], x["v"].shape[2]))
    if heads is not None:
        S0 = S0[:, heads]
    dsf = None if d_sf is None else _np(d_sf)
    if dsf is not None and heads is not None:
        dsf = dsf[:, heads]
    return oracle.kda_backward(q, k, v, g, b, S0, x["cu_seqlens"].cpu().numpy(),
                               sel(_np(d_out)), dsf)


@pytest.mark.parametrize("act,dk,dv,lengths,slow", [
    ("f32", 32, 32, [100, 37], True),
    ("f32", 48, 40, [53, 0, 81, 16], True),   # ragged column block (40 = 32 + 8)
    ("f32", 16, 16, [64], False),
    ("bf16", 128, 128, [70, 33], True),
    ("bf16", 128, 96, [47, 90], False),
    # rows that are not whole 16-byte units: the producer's plain-load path
    ("f32", 30, 20, [45, 19], True),
    ("bf16", 60, 44, [33, 70], False),
])
def test_backward_matches_oracle(act, dk, dv, lengths, slow):
    H = 2
    x = make_prefill_inputs(lengths, H, dk, dv, act, s0_std=1.0, seed=31, slow_decay=slow)
    d_out, d_sf = make_backward_adjoints(sum(lengths), len(lengths), H, dk, dv, act, seed=32)
    got = _run(x, d_out, d_sf)
    ref = _oracle(x, d_out, d_sf)
    for name, a, b in zip(NAMES, got, ref):
        assert rel_err(_np(a), b) <= _tol(act, dk, dv), (name, rel_err(_np(a), b))


@pytest.mark.parametrize("act,d,lengths,nseg", [
    ("f32", 32, [300, 77, 0, 129], 2),
    ("f32", 32, [300, 77, 0, 129], 5),
    ("f32", 48, [200, 31], 3),
    ("bf16", 128, [250, 90], 4),
    ("bf16", 128, [250, 90], 0),    # the library's choice
    ("bf16", 128, [700, 0, 333, 45], 16),  # chunked: empty sequence, more segments
    ("bf16", 128, [40, 5, 0], 8),   # chunked: segments without a block
    ("bf16", 60, [100, 45], 3),     # plain-load producer
    ("f32", 16, [40, 5, 0], 8),     # more segments than 16-token chunks: empty segments
    ("f32", 32, [1500, 260], 64),   # the largest split
])
def test_backward_segments_match_oracle(act, d, lengths, nseg):
    """The segment split (per-segment transfer matrices, zero-start states and
    zero-end adjoints, fp32 scans, then the gradient pass per segment) against the
    oracle, with a material initial state and final-state adjoint (slow decay)."""
    H = 2
    x = make_prefill_inputs(lengths, H, d, d, act, s0_std=1.0, seed=41, slow_decay=True)
    d_out, d_sf = make_backward_adjoints(sum(lengths), len(lengths), H, d, d, act, seed=42)
    got = _run(x, d_out, d_sf, num_segments=nseg)
    ref = _oracle(x, d_out, d_sf)
    for name, a, b in zip(NAMES, got, ref):
        assert rel_err(_np(a), b) <= _tol(act, d, d), (name, rel_err(_np(a), b))


@pytest.mark.parametrize("act,d", [("f32", 32), ("bf16", 128)])
def test_backward_without_initial_or_final_state(act, d):
    lengths = [29, 0, 50]
    x = make_prefill_inputs(lengths, 2, d, d, act, seed=33)
    d_out, _ = make_backward_adjoints(sum(lengths), 3, 2, d, d, act, seed=34, final=False)
    got = _run(x, d_out, None)
    ref = _oracle(x, d_out, None)  # zero S0: its gradient is still defined
    for name, a, b in zip(NAMES, got, ref):
        assert rel_err(_np(a), b) <= _tol(act, d, d), name
    # an empty sequence's dS0 is its (zero) final-state adjoint
    assert torch.count_nonzero(got[5][1]) == 0


def test_backward_skips_dS0_and_overwrites_outputs():
    lengths = [40, 24]
    x = make_prefill_inputs(lengths, 2, 32, 32, "f32", s0_std=1.0, seed=35)
    d_out, d_sf = make_backward_adjoints(64, 2, 2, 32, 32, "f32", seed=36)
    a = _run(x, d_out, d_sf)
    b = _run(x, d_out, d_sf, want_dS0=False)
    assert b[5] is None
    for u, w in zip(a[:5], b[:5]):  # the accumulated outputs start from zero every call
        assert torch.allclose(u, w, rtol=0, atol=1e-6 * float(u.abs().max()))


def test_backward_bench_size_sampled_heads_and_linearity():
    """B=1, H=8, T=4096, d=128 BF16 (the bench workload): heads 0 and 5 against the
    oracle; all heads: the gradients are linear in (d_out, d_S_final)."""
    T, H, d = 4096, 8, 128
    x = make_prefill_inputs([T], H, d, d, "bf16", seed=37)
    d1, s1 = make_backward_adjoints(T, 1, H, d, d, "bf16", seed=38)
    got = _run(x, d1, s1)
    for h in (0, 5):
        ref = _oracle(x, d1, s1, heads=[h])
        for name, a, b in zip(NAMES, got, ref):
            a = _np(a)[:, [h]]
            assert rel_err(a, b) <= _tol("bf16", d, d), (h, name, rel_err(a, b))
    # linearity: backward(2 d_out, 2 d_S_final) = 2 backward(d_out, d_S_final),
    # exact in binary floating point (scaling by 2 commutes with every rounding)
    g2 = _run(x, (d1.float() * 2).to(d1.dtype), s1 * 2)
    for name, a, b in zip(NAMES, got, g2):
        assert rel_err(_np(b), 2 * _np(a)) <= 1e-5, name


def test_backward_unaligned_inputs_take_the_plain_path():
    """Inputs one fp32 element past a 16-byte boundary (the entry point needs 4-byte
    alignment only): same gradients as the oracle."""
    lengths = [37, 52]
    H, d = 2, 32
    x = make_prefill_inputs(lengths, H, d, d, "f32", s0_std=1.0, seed=39, slow_decay=True)
    d_out, d_sf = make_backward_adjoints(sum(lengths), 2, H, d, d, "f32", seed=40)

    def shifted(t):  # the same values at a device address 4 bytes past 16-byte alignment
        buf = torch.empty(t.numel() + 4, dtype=t.dtype, device="cuda")
        view = buf[1:1 + t.numel()].view(t.shape)
        view.copy_(t.cuda())
        assert view.data_ptr() % 16 == 4
        return view

    got = kda.prefill_backward(shifted(x["q"]), shifted(x["k"]), shifted(x["v"]), shifted(x["g"]),
                               x["beta"].cuda(), x["S0"].cuda(), x["cu_seqlens"].cuda(),
                               shifted(d_out), d_sf.cuda())
    torch.cuda.synchronize()
    ref = _oracle(x, d_out, d_sf)
    for name, a, b in zip(NAMES, got, ref):
        assert rel_err(_np(a), b) <= TOL, name


@pytest.mark.parametrize("act,d", [("f32", 32), ("bf16", 128)])
def test_autograd_function_gradients(act, d):
    """kda_prefill as a torch.autograd.Function: .grad of every input after
    loss = <d_out, o> + <d_S_final, S_final> against the oracle (BF16 inputs get
    BF16 gradients, so their bound is the BF16 one)."""
    from kimi_delta_attention_18_gb300.autograd import kda_prefill
    lengths = [90, 41]
    H = 2
    x = make_prefill_inputs(lengths, H, d, d, act, s0_std=1.0, seed=43, slow_decay=True)
    d_out, d_sf = make_backward_adjoints(sum(lengths), 2, H, d, d, act, seed=44)
    leaves = {n: x[n].cuda().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "S0")}
    o, SF = kda_prefill(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                        leaves["S0"], x["cu_seqlens"].cuda())
    loss = (o.float() * d_out.cuda().float()).sum() + (SF * d_sf.cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    ref = _oracle(x, d_out, d_sf)
    tol = 1e-4 if act == "f32" else 2e-2
    for name, leaf, b in zip(NAMES, ("q", "k", "v", "g", "beta", "S0"), ref):
        got = leaves[leaf].grad
        assert got.dtype == leaves[leaf].dtype
        assert rel_err(_np(got), b) <= tol, (name, rel_err(_np(got), b))


def test_backward_piecewise_equals_whole():
    """A sequence differentiated in two pieces, last piece first, each from its
    start state with d_S_final = the next piece's dS0 (the documented use for
    batches whose workspace does not fit), against the oracle on the whole."""
    L, cut, H, d = 300, 130, 2, 32
    x = make_prefill_inputs([L], H, d, d, "f32", s0_std=1.0, seed=45, slow_decay=True)
    d_out, d_sf = make_backward_adjoints(L, 1, H, d, d, "f32", seed=46)
    c = {n: x[n].cuda() for n in ("q", "k", "v", "g", "beta", "S0")}
    dO, dSF = d_out.cuda(), d_sf.cuda()
    one = lambda n: torch.tensor([0, n], dtype=torch.int32, device="cuda")
    p1 = {n: t[:cut].contiguous() for n, t in c.items() if n != "S0"}
    p2 = {n: t[cut:].contiguous() for n, t in c.items() if n != "S0"}
    _, S_mid = kda.prefill_chunked(p1["q"], p1["k"], p1["v"], p1["g"], p1["beta"], c["S0"],
                                   one(cut))
    g2 = kda.prefill_backward(p2["q"], p2["k"], p2["v"], p2["g"], p2["beta"], S_mid,
                              one(L - cut), dO[cut:].contiguous(), dSF)
    g1 = kda.prefill_backward(p1["q"], p1["k"], p1["v"], p1["g"], p1["beta"], c["S0"], one(cut),
                              dO[:cut].contiguous(), g2[5])
    torch.cuda.synchronize()
    ref = _oracle(x, d_out, d_sf)
    for i, name in enumerate(NAMES[:5]):
        got = torch.cat([g1[i], g2[i]], dim=0)
        assert rel_err(_np(got), ref[i]) <= TOL, name
    assert rel_err(_np(g1[5]), ref[5]) <= TOL
