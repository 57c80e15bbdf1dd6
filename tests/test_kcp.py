"""KCP across ranks (kimi_delta_attention_18_gb300.kcp) on the CPU: the exchange
and the bookkeeping around the three compute steps, with the oracle standing in
for the kernels.  W ranks emulated in one process, and real 2- and 3-rank gloo
process groups (all_gather of the fixed-size (A, B) pairs), both against the
oracle's whole-batch recurrence."""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from kimi_delta_attention_18_gb300 import kcp
from kimi_delta_attention_18_gb300.inputs import make_prefill_inputs

LENGTHS = [150, 37, 0, 64]
H, D = 2, 8


def _inputs():
    x = make_prefill_inputs(LENGTHS, H, D, D, "f32", s0_std=1.0, seed=51, slow_decay=True)
    return {n: (t.double() if isinstance(t, torch.Tensor) and t.is_floating_point() else t)
            for n, t in x.items()}


def oracle_ops():
    def transfer(k, v, g, beta, cu, W, r):
        A, B = oracle.kda_state_transfer(k.numpy(), v.numpy(), g.numpy(), beta.numpy(),
                                         cu.numpy(), W)
        return torch.from_numpy(A[:, :, r].copy()), torch.from_numpy(B[:, :, r].copy())

    def compose(A, B, S0):
        st, sf = oracle.kda_state_compose(A.numpy(), B.numpy(),
                                          None if S0 is None else S0.numpy())
        return torch.from_numpy(st), torch.from_numpy(sf)

    def segment(q, k, v, g, beta, starts, cu, W, r):
        bounds = oracle.segment_bounds(cu.numpy(), W)
        out = np.zeros((q.shape[0], q.shape[1], v.shape[2]))
        for n in range(bounds.shape[0]):
            a, b = (int(t) for t in bounds[n, r])
            if b > a:
                o, _ = oracle.kda_forward(q[a:b].numpy(), k[a:b].numpy(), v[a:b].numpy(),
                                          g[a:b].numpy(), beta[a:b].numpy(),
                                          starts[n, :, r].numpy()[None],
                                          np.array([0, b - a], dtype=np.int32))
                out[a:b] = o
        return torch.from_numpy(out)

    return kcp.KCPOps(transfer, compose, segment)


def _reference(x):
    return oracle.kda_forward(*(x[n].numpy() for n in ("q", "k", "v", "g", "beta")),
                              x["S0"].numpy(), x["cu_seqlens"].numpy())


def _check(x, outs, finals, W):
    o_ref, S_ref = _reference(x)
    T = x["q"].shape[0]
    total = torch.zeros_like(torch.from_numpy(o_ref))
    cover = torch.zeros(T, dtype=torch.int64)
    for r in range(W):
        m = kcp.segment_token_mask(x["cu_seqlens"], W, r, T)
        cover += m.long()
        assert torch.count_nonzero(outs[r][~m]) == 0  # a rank writes its own tokens only
        total += outs[r]
    assert torch.all(cover == 1)  # the segments partition the tokens
    scale = float(np.abs(o_ref).max())
    assert float((total - torch.from_numpy(o_ref)).abs().max()) <= 1e-10 * scale
    for f in finals:
        assert np.abs(f.numpy() - S_ref).max() <= 1e-10 * np.abs(S_ref).max()


def test_segment_mask_is_the_transfer_split():
    cu = torch.tensor([0, 150, 187, 187, 251], dtype=torch.int32)
    for W in (1, 2, 3, 7):
        b = oracle.segment_bounds(cu.numpy(), W)
        for r in range(W):
            m = kcp.segment_token_mask(cu, W, r, 251)
            ref = np.zeros(251, dtype=bool)
            for n in range(b.shape[0]):
                ref[b[n, r, 0]:b[n, r, 1]] = True
            assert np.array_equal(m.numpy(), ref)


@pytest.mark.parametrize("W", [1, 2, 3, 5])
def test_kcp_emulated_ranks(W):
    x = _inputs()
    ops = oracle_ops()
    args = (x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"])
    pairs = [kcp.local_pairs(*args, W, r, ops) for r in range(W)]
    A_all = torch.stack([p[0] for p in pairs], dim=2)
    B_all = torch.stack([p[1] for p in pairs], dim=2)
    res = [kcp.finish(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["cu_seqlens"], W, r,
                      A_all, B_all, ops) for r in range(W)]
    _check(x, [o for o, _ in res], [f for _, f in res], W)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, path):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        x = _inputs()
        out, S_final = kcp.kcp_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"],
                                       x["cu_seqlens"], ops=oracle_ops())
        torch.save({"out": out, "S_final": S_final}, os.path.join(path, "rank%d.pt" % rank))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_kcp_gloo_all_gather(world):
    with tempfile.TemporaryDirectory() as path:
        mp.spawn(_rank_main, args=(world, _free_port(), path), nprocs=world, join=True)
        res = [torch.load(os.path.join(path, "rank%d.pt" % r)) for r in range(world)]
    _check(_inputs(), [r["out"] for r in res], [r["S_final"] for r in res], world)


def test_default_steps_need_the_gpu_library():
    """The default steps are libkda's: on CPU tensors they raise, no fallback."""
    x = _inputs()
    f = {n: x[n].float() for n in ("k", "v", "g", "beta")}
    with pytest.raises((ValueError, RuntimeError, OSError)):
        kcp.local_pairs(f["k"], f["v"], f["g"], f["beta"], x["cu_seqlens"], 2, 0)


def test_check_catches_a_wrong_start_state():
    """A rank that runs its segment from its neighbour's start state (a plausible
    off-by-one in the scan bookkeeping, planted in the oracle-backed steps) fails
    the comparison."""
    x = _inputs()
    good = oracle_ops()

    def shifted_segment(q, k, v, g, beta, starts, cu, W, r):  # segment r from start r - 1
        return good.segment(q, k, v, g, beta, torch.roll(starts, 1, dims=2), cu, W, r)

    bad = kcp.KCPOps(good.transfer, good.compose, shifted_segment)
    W = 3
    args = (x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"])
    pairs = [kcp.local_pairs(*args, W, r, bad) for r in range(W)]
    A_all = torch.stack([p[0] for p in pairs], dim=2)
    B_all = torch.stack([p[1] for p in pairs], dim=2)
    res = [kcp.finish(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["cu_seqlens"], W, r,
                      A_all, B_all, bad) for r in range(W)]
    with pytest.raises(AssertionError):
        _check(x, [o for o, _ in res], [f for _, f in res], W)
