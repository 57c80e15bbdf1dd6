"""Pins for the fp64 oracle: each test checks it against something other than
itself -- brute-force matrix products, closed forms, special cases that reduce
to textbook recurrences, invariants -- chosen so that a dropped term, a wrong
sign, a wrong index or a swapped order of operations fails at least one.

Sources: "Kimi K3 Architecture Explained", section 3 (lineage linear attention
-> DeltaNet -> Gated DeltaNet -> KDA; decay, then erase, then write) and the
Kimi K3 technical-report digest, sections 2.1 (1) (channel-wise gate, g_min = -5,
16-token blocks in BF16 range) and 2.4 (1) (transfer matrix + zero-initial
state, prefix scan).
"""
import numpy as np
import pytest

import oracle
from oracle.chunked import kda_forward_chunked
from tests.conftest import rel_err


def _rand(rng, T, H, dk, dv, unit_k=True, s0=True, g_scale=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -5.0 / (1.0 + np.exp(-g_scale * rng.standard_normal((T, H, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = rng.standard_normal((1, H, dk, dv)) if s0 else None
    return q, k, v, g, beta, S0


def _dense_reference(q, k, v, g, beta, S0, order="decay_first"):
    """Brute force: build every step as explicit d x d matrices."""
    T, H, dk = k.shape
    dv = v.shape[2]
    out = np.zeros((T, H, dv))
    SF = np.zeros((1, H, dk, dv))
    for h in range(H):
        S = np.zeros((dk, dv)) if S0 is None else S0[0, h].copy()
        for t in range(T):
            D = np.diag(np.exp(g[t, h]))
            E = np.eye(dk) - beta[t, h] * np.outer(k[t, h], k[t, h])
            Wr = beta[t, h] * np.outer(k[t, h], v[t, h])
            if order == "decay_first":
                S = E @ (D @ S) + Wr
            else:  # erase first, then decay
                S = D @ (E @ S) + Wr
            out[t, h] = S.T @ q[t, h]
        SF[0, h] = S
    return out, SF


@pytest.mark.parametrize("d,T", [(2, 5), (4, 8), (16, 7)])
def test_matches_dense_matrix_products(d, T):
    rng = np.random.default_rng(d * 100 + T)
    q, k, v, g, beta, S0 = _rand(rng, T, 2, d, d)
    o, S = oracle.kda_forward(q, k, v, g, beta, S0)
    o_ref, S_ref = _dense_reference(q, k, v, g, beta, S0)
    assert rel_err(o, o_ref) < 1e-13
    assert rel_err(S, S_ref) < 1e-13


def test_order_is_decay_then_erase():
    """With a per-channel (non-scalar) decay the two orders differ; the oracle must
    follow decay-then-erase (page 1, section 3) and differ from the other order."""
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = _rand(rng, 4, 1, 2, 2)
    g[..., 0] = -0.1
    g[..., 1] = -3.0
    o, S = oracle.kda_forward(q, k, v, g, beta, S0)
    o_df, S_df = _dense_reference(q, k, v, g, beta, S0, "decay_first")
    o_ef, S_ef = _dense_reference(q, k, v, g, beta, S0, "erase_first")
    assert rel_err(S, S_df) < 1e-13
    assert rel_err(S_df, S_ef) > 1e-2
    assert rel_err(S, S_ef) > 1e-2


def test_deltanet_recall_compare_write_form():
    """DeltaNet reading (page 1, section 3): recall with the key, compare with the new
    value, write the difference: S' = DS + beta k (v - (DS)^T k)^T."""
    rng = np.random.default_rng(3)
    dk, dv = 8, 5
    q, k, v, g, beta, S0 = _rand(rng, 1, 1, dk, dv)
    _, S = oracle.kda_forward(q, k, v, g, beta, S0)
    DS = np.exp(g[0, 0])[:, None] * S0[0, 0]
    recalled = DS.T @ k[0, 0]
    expect = DS + beta[0, 0] * np.outer(k[0, 0], v[0, 0] - recalled)
    assert rel_err(S[0, 0], expect) < 1e-13


def test_exact_recall_with_unit_key():
    """No decay, beta = 1, a unit key: after the step the state recalls exactly v for
    that key; for beta < 1 it recalls (1 - beta) (DS)^T k + beta v."""
    rng = np.random.default_rng(11)
    dk, dv = 6, 4
    S0 = rng.standard_normal((1, 1, dk, dv))
    k = rng.standard_normal((1, 1, dk)); k /= np.linalg.norm(k)
    v = rng.standard_normal((1, 1, dv))
    q = k.copy()
    _, S = oracle.kda_forward(q, k, v, np.zeros((1, 1, dk)), np.ones((1, 1)), S0)
    np.testing.assert_allclose(S[0, 0].T @ k[0, 0], v[0, 0], rtol=0, atol=1e-13)
    g = -rng.uniform(0, 5, (1, 1, dk))
    b = 0.3
    _, S = oracle.kda_forward(q, k, v, g, np.full((1, 1), b), S0)
    DS = np.exp(g[0, 0])[:, None] * S0[0, 0]
    np.testing.assert_allclose(S[0, 0].T @ k[0, 0], (1 - b) * DS.T @ k[0, 0] + b * v[0, 0],
                               rtol=0, atol=1e-13)


def test_beta_zero_is_pure_decay():
    """beta = 0 read literally: nothing is erased or written, so S_t = P_t S0 with
    P_t = Diag(exp(g_1 + ... + g_t)) and o_t = (P_t S0)^T q_t; from S0 = 0 all is 0."""
    rng = np.random.default_rng(5)
    T, H, dk, dv = 9, 2, 5, 3
    q, k, v, g, beta, S0 = _rand(rng, T, H, dk, dv)
    beta[:] = 0.0
    o, S = oracle.kda_forward(q, k, v, g, beta, S0)
    G = np.cumsum(g, axis=0)
    for h in range(H):
        for t in range(T):
            St = np.exp(G[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(S[0, h], np.exp(G[-1, h])[:, None] * S0[0, h], rtol=1e-13)
    o0, S0out = oracle.kda_forward(q, k, v, g, beta, None)
    assert np.all(o0 == 0.0) and np.all(S0out == 0.0)


def _gla_parallel(q, k, v, g, beta, S0):
    """Gated linear attention in its quadratic (attention-matrix) form:
    o_t = sum_{i<=t} ((q_t * exp(G_t - G_i)) . k_i) beta_i v_i + (P_t S0)^T q_t."""
    T, H, dk = k.shape
    G = np.cumsum(g, axis=0)
    out = np.zeros((T, H, v.shape[2]))
    for h in range(H):
        for t in range(T):
            acc = np.zeros(v.shape[2])
            for i in range(t + 1):
                w = np.sum(q[t, h] * np.exp(G[t, h] - G[i, h]) * k[i, h])
                acc += w * beta[i, h] * v[i, h]
            if S0 is not None:
                acc += (np.exp(G[t, h])[:, None] * S0[0, h]).T @ q[t, h]
            out[t, h] = acc
    return out


def test_erase_off_is_gated_linear_attention():
    rng = np.random.default_rng(9)
    q, k, v, g, beta, S0 = _rand(rng, 12, 2, 6, 4)
    o, _ = oracle.kda_forward(q, k, v, g, beta, S0, erase=False)
    assert rel_err(o, _gla_parallel(q, k, v, g, beta, S0)) < 1e-12


def test_erase_off_no_decay_is_linear_attention():
    rng = np.random.default_rng(10)
    T, H, dk, dv = 10, 1, 4, 3
    q, k, v, g, beta, S0 = _rand(rng, T, H, dk, dv)
    g[:] = 0.0
    o, S = oracle.kda_forward(q, k, v, g, beta, S0, erase=False)
    A = np.tril(q[:, 0] @ k[:, 0].T)               # causal q.k scores
    expect = A @ (beta[:, 0:1] * v[:, 0]) + q[:, 0] @ S0[0, 0]
    assert rel_err(o[:, 0], expect) < 1e-13
    assert rel_err(S[0, 0], S0[0, 0] + k[:, 0].T @ (beta[:, 0:1] * v[:, 0])) < 1e-13


def test_scalar_decay_is_gated_deltanet():
    """One decay value shared by all channels (Gated DeltaNet, page 1 section 3):
    decay and erase then commute, so S_t = alpha_t (I - beta k k^T) S + beta k v^T."""
    rng = np.random.default_rng(12)
    T, H, dk, dv = 8, 2, 5, 4
    q, k, v, g, beta, S0 = _rand(rng, T, H, dk, dv)
    g[:] = g[:, :, :1]
    o, S = oracle.kda_forward(q, k, v, g, beta, S0)
    for h in range(H):
        St = S0[0, h].copy()
        for t in range(T):
            a = np.exp(g[t, h, 0])
            St = a * (St - beta[t, h] * np.outer(k[t, h], k[t, h] @ St)) + \
                beta[t, h] * np.outer(k[t, h], v[t, h])
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-12, atol=1e-13)


def test_scalar_geometric_closed_form():
    """d = 1, constant alpha, beta, k = 1, v = c: s_t = a s_{t-1} + beta c with
    a = (1 - beta) alpha, so s_t = a^t s0 + beta c (1 - a^t) / (1 - a)."""
    T, alpha, b, c, s0 = 20, np.exp(-0.7), 0.35, 1.7, -0.4
    ones = np.ones((T, 1, 1))
    o, S = oracle.kda_forward(ones, ones, c * ones, np.full((T, 1, 1), np.log(alpha)),
                              np.full((T, 1), b), np.full((1, 1, 1, 1), s0))
    a = (1 - b) * alpha
    t = np.arange(1, T + 1)
    expect = a ** t * s0 + b * c * (1 - a ** t) / (1 - a)
    np.testing.assert_allclose(o[:, 0, 0], expect, rtol=1e-13)
    np.testing.assert_allclose(S[0, 0, 0, 0], expect[-1], rtol=1e-13)


def test_linearity_in_initial_state_and_values():
    """For fixed (q, k, g, beta) the map (S0, V) -> (O, S_T) is linear; this is what
    the transfer-matrix / zero-initial-state split rests on."""
    rng = np.random.default_rng(13)
    q, k, v, g, beta, S0 = _rand(rng, 11, 2, 6, 5)
    o, S = oracle.kda_forward(q, k, v, g, beta, S0)
    o1, S1 = oracle.kda_forward(q, k, np.zeros_like(v), g, beta, S0)
    o2, S2 = oracle.kda_forward(q, k, v, g, beta, None)
    assert rel_err(o, o1 + o2) < 1e-13
    assert rel_err(S, S1 + S2) < 1e-13


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_chunked_wy_form_matches_recurrence(C):
    """The chunked WY/UT form (16-token blocks on the pages; any block size in exact
    arithmetic), including partial last chunks and packed sequences."""
    rng = np.random.default_rng(20 + C)
    lengths = [37, 16, 5, 0, 50]
    T = sum(lengths)
    q, k, v, g, beta, _ = _rand(rng, T, 2, 8, 6)
    S0 = rng.standard_normal((len(lengths), 2, 8, 6))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S = oracle.kda_forward(q, k, v, g, beta, S0, cu)
    oc, Sc = kda_forward_chunked(q, k, v, g, beta, S0, cu, chunk=C)
    assert rel_err(oc, o) < 1e-12
    assert rel_err(Sc, S) < 1e-12


def test_block_exponent_range_bound():
    """g = -5 sigmoid(x) lies in (-5, 0), so over a 16-token block |Gamma| < 80, and
    exp(+-80) stays inside the BF16/fp32 normal range (ln max ~ 88.7,
    ln min-normal ~ -87.3): digest section 2.1 (1)."""
    import torch
    from kimi_delta_attention_18_gb300.inputs import make_prefill_inputs
    x = make_prefill_inputs([4096], 8, 128, 128, "bf16", seed=0)
    g = x["g"].double().numpy()
    assert g.max() < 0.0 and g.min() > -5.0
    Gam = np.cumsum(g.reshape(256, 16, 8, 128), axis=1)
    assert np.abs(Gam).max() < 80.0
    assert 80.0 < np.log(float(torch.finfo(torch.bfloat16).max))
    assert -80.0 > np.log(float(torch.finfo(torch.bfloat16).tiny))


def test_state_norm_never_grows_faster_than_the_write():
    """Unit keys, beta in [0,1], alpha <= 1: ||I - beta k k^T|| <= 1 and ||Diag(alpha)||
    <= 1, so ||S_t||_2 <= ||S_{t-1}||_2 + beta ||v_t||."""
    rng = np.random.default_rng(17)
    T, dk, dv = 30, 8, 8
    q, k, v, g, beta, S0 = _rand(rng, T, 1, dk, dv)
    S = S0[0]
    for t in range(T):
        _, S_new = oracle.kda_decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                          beta[t:t + 1], S[None])
        S_new = S_new[0]
        lhs = np.linalg.norm(S_new[0], 2)
        rhs = np.linalg.norm(S[0], 2) + beta[t, 0] * np.linalg.norm(v[t, 0])
        assert lhs <= rhs * (1 + 1e-12)
        S = S_new


def test_resume_and_decode_continue_the_same_sequence():
    """Prefix caching: a state saved after a tokens and fed back as S0 continues the
    sequence exactly (digest section 2.4 (4): the KDA state is the cache unit);
    decode steps continue a prefill exactly."""
    rng = np.random.default_rng(19)
    T, a = 29, 13
    q, k, v, g, beta, S0 = _rand(rng, T, 3, 6, 5)
    o, S = oracle.kda_forward(q, k, v, g, beta, S0)
    oa, Sa = oracle.kda_forward(q[:a], k[:a], v[:a], g[:a], beta[:a], S0)
    ob, Sb = oracle.kda_forward(q[a:], k[a:], v[a:], g[a:], beta[a:], Sa)
    assert rel_err(np.concatenate([oa, ob]), o) < 1e-13 and rel_err(Sb, S) < 1e-13
    od, Sd = oracle.kda_decode_step(q[a][None], k[a][None], v[a][None], g[a][None],
                                    beta[a][None], Sa)
    assert rel_err(od[0], o[a]) < 1e-13
    _, Sa1 = oracle.kda_forward(q[:a + 1], k[:a + 1], v[:a + 1], g[:a + 1], beta[:a + 1], S0)
    assert rel_err(Sd, Sa1) < 1e-13


def test_packing_equals_separate_sequences():
    rng = np.random.default_rng(21)
    lengths = [7, 0, 19, 3]
    T = sum(lengths)
    q, k, v, g, beta, _ = _rand(rng, T, 2, 4, 4)
    S0 = rng.standard_normal((4, 2, 4, 4))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S = oracle.kda_forward(q, k, v, g, beta, S0, cu)
    for n in range(4):
        a, b = cu[n], cu[n + 1]
        on, Sn = oracle.kda_forward(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], S0[n:n + 1])
        if b > a:
            assert rel_err(o[a:b], on) < 1e-14
        assert rel_err(S[n], Sn[0]) < 1e-14


def test_threading_and_column_split_are_exact():
    rng = np.random.default_rng(23)
    q, k, v, g, beta, S0 = _rand(rng, 40, 3, 16, 16)
    o1, S1 = oracle.kda_forward(q, k, v, g, beta, S0, threads=1, col_block=16)
    o2, S2 = oracle.kda_forward(q, k, v, g, beta, S0, threads=4, col_block=3)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


@pytest.mark.parametrize("nseg", [1, 4, 7])
def test_transfer_matrix_and_zero_state_split(nseg):
    """Digest section 2.4 (1): per segment, S_end = A S_start + B; the compositions
    are associative; a scan over segments reproduces the sequential state."""
    rng = np.random.default_rng(30 + nseg)
    lengths = [100, 33]
    T = sum(lengths)
    q, k, v, g, beta, _ = _rand(rng, T, 2, 6, 5, g_scale=0.2)
    g *= 0.001  # slow forgetting, so the transfer matrices stay material
    beta *= 0.1
    S0 = rng.standard_normal((2, 2, 6, 5))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    A, B = oracle.kda_state_transfer(k, v, g, beta, cu, nseg)
    bounds = oracle.segment_bounds(cu, nseg)
    # S_end = A S_start + B for a random start state, segment by segment
    for n in range(2):
        for s in range(nseg):
            a, b = bounds[n, s]
            Sst = rng.standard_normal((1, 2, 6, 5))
            _, Se = oracle.kda_forward(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], Sst)
            for h in range(2):
                assert rel_err(A[n, h, s] @ Sst[0, h] + B[n, h, s], Se[0, h]) < 1e-12
    assert np.abs(A).max() > 0.1  # not trivially forgotten
    # scan reproduces the sequential final state and per-segment start states
    starts, SF = oracle.kda_state_compose(A.reshape(4, nseg, 6, 6), B.reshape(4, nseg, 6, 5),
                                          S0.reshape(4, 6, 5))
    _, S_seq = oracle.kda_forward(q, k, v, g, beta, S0, cu)
    assert rel_err(SF.reshape(2, 2, 6, 5), S_seq) < 1e-12
    if nseg > 1:
        # associativity: (A2,B2) o (A1,B1) = (A2 A1, A2 B1 + B2) equals the merged segment
        A2, B2 = oracle.kda_state_transfer(k, v, g, beta, cu, 1)
        Aacc = np.broadcast_to(np.eye(6), (2, 2, 6, 6)).copy()
        Bacc = np.zeros((2, 2, 6, 5))
        for s in range(nseg):
            Bacc = A[:, :, s] @ Bacc + B[:, :, s]
            Aacc = A[:, :, s] @ Aacc
        assert rel_err(Aacc, A2[:, :, 0]) < 1e-12
        assert rel_err(Bacc, B2[:, :, 0]) < 1e-12


def test_segment_bounds_cover_each_sequence_once():
    cu = np.array([0, 100, 100, 133, 149])
    for nseg in (1, 3, 8, 64):
        b = oracle.segment_bounds(cu, nseg)
        for n in range(4):
            assert b[n, 0, 0] == cu[n] and b[n, -1, 1] == cu[n + 1]
            assert np.all(b[n, 1:, 0] == b[n, :-1, 1])
            assert np.all((b[n, :, 0] - cu[n]) % 16 == 0)


def test_gate_prologue_closed_forms():
    """g = -5 sigmoid(x) and beta = sigmoid(x) at points with exact values, the
    reflection sigmoid(x) + sigmoid(-x) = 1 (catches a sign slip in the
    exponent), and the per-row L2 normalisation of q and k (3-4-5 rows, a zero
    row, scale invariance, over the last axis only)."""
    x = np.array([0.0, np.log(3.0), -np.log(3.0), 40.0, -40.0])
    q = np.array([[[3.0, 4.0]], [[0.0, 0.0]], [[-6.0, 8.0]]])  # [T=3, H=1, d=2]
    k = 2.5 * q
    qn, kn, g, beta = oracle.gate_prologue(q, k, x, x)
    assert g[0] == -2.5 and beta[0] == 0.5
    assert abs(beta[1] - 0.75) < 1e-15 and abs(beta[2] - 0.25) < 1e-15
    assert abs(g[1] + 3.75) < 1e-14 and abs(g[2] + 1.25) < 1e-14
    assert abs(g[3] + 5.0) < 1e-15 and -1e-15 < g[4] < 0.0
    assert np.allclose(g[[1, 3]] + g[[2, 4]], -5.0, atol=1e-14, rtol=0)
    assert np.allclose(qn[0, 0], [0.6, 0.8], atol=1e-15) and np.all(qn[1] == 0.0)
    assert np.allclose(qn[2, 0], [-0.6, 0.8], atol=1e-15)
    assert np.allclose(kn, qn, atol=1e-15)  # scale invariance
    rows = oracle.gate_prologue(np.random.default_rng(1).normal(size=(5, 3, 16)),
                                np.zeros((5, 3, 16)), np.zeros(1), np.zeros(1))[0]
    assert np.allclose(np.linalg.norm(rows, axis=-1), 1.0, atol=1e-14)


def test_backward_forward_matches_and_finite_differences():
    """The backward's own forward equals the C oracle, and every gradient equals
    central finite differences of the C oracle's loss on a tiny problem (two
    sequences, S0, non-uniform gates), so a dropped term or a wrong sign in the
    differentiated loop fails here and not only on the GPU."""
    rng = np.random.default_rng(7)
    lengths, H, d = [4, 3], 2, 3
    T = sum(lengths)
    cu = np.array([0, 4, 7], dtype=np.int32)
    q, k, v = (rng.normal(size=(T, H, d)) for _ in range(3))
    g = -5.0 / (1.0 + np.exp(-rng.normal(size=(T, H, d))))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=(T, H))))
    S0 = rng.normal(size=(2, H, d, d))
    dO = rng.normal(size=(T, H, d))
    dSF = rng.normal(size=(2, H, d, d))
    grads = oracle.kda_backward(q, k, v, g, beta, S0, cu, dO, dSF)

    def loss(q_, k_, v_, g_, b_, s_):
        o, sf = oracle.kda_forward(q_, k_, v_, g_, b_, s_, cu)
        return float(np.sum(o * dO) + np.sum(sf * dSF))

    args = [q, k, v, g, beta, S0]
    eps = 1e-6
    for which, grad in enumerate(grads):
        x = args[which]
        flat = x.reshape(-1)
        fd = np.zeros_like(flat)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            up = loss(*args)
            flat[i] = keep - eps
            dn = loss(*args)
            flat[i] = keep
            fd[i] = (up - dn) / (2 * eps)
        assert np.allclose(grad.reshape(-1), fd, rtol=1e-6, atol=1e-7), which


@pytest.mark.parametrize("chunk", [1, 5, 16])
@pytest.mark.parametrize("slow", [False, True])
def test_chunked_backward_equals_token_backward(chunk, slow):
    """The chunk-level adjoint (oracle/chunked.py: through the UT transform's
    inverse, the masked in-chunk products and the cumulative log-decay) gives the
    autograd gradients of the token recurrence, for any chunk size, ragged
    sequences included."""
    from oracle import chunked
    from kimi_delta_attention_18_gb300.inputs import make_backward_adjoints, make_prefill_inputs
    lengths = [37, 20, 0, 16]
    x = make_prefill_inputs(lengths, 2, 6, 5, "f32", seed=61, s0_std=1.0, slow_decay=slow)
    d_out, d_sf = make_backward_adjoints(sum(lengths), len(lengths), 2, 6, 5, "f32", seed=62)
    f = lambda t: t.double().numpy()
    args = [f(x[n]) for n in ("q", "k", "v", "g", "beta", "S0")]
    cu = x["cu_seqlens"].numpy()
    ref = oracle.kda_backward(*args, cu, f(d_out), f(d_sf))
    got = chunked.kda_backward_chunked(*args, cu, f(d_out), f(d_sf), chunk=chunk)
    for a, b in zip(got, ref):
        assert np.abs(a - b).max() <= 1e-12 * max(np.abs(b).max(), 1e-300)
