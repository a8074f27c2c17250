"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

None of these compares the oracle with itself. They use the pages' worked numbers
(tests/golden/toy_traces.json), closed forms, the textbook delta rule, brute-force products of
the transition matrices M_t, and invariants. Together they catch a dropped term, a wrong sign
or index, a transposed operand, a decay applied after instead of before the write, or an output
read from the pre-update state.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import chunkwise as cw

RNG = np.random.default_rng(1234)


def _rand_inputs(B, T, H, dk, dv, rng, g_lo=-5.0, unit=True, beta_lo=0.0, beta_hi=1.0):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    g = rng.uniform(g_lo, 0.0, (B, T, H, dk))
    beta = rng.uniform(beta_lo, beta_hi, (B, T, H))
    return q, k, v, g, beta


def _one_head(x):
    return x[None, :, None]


# ---------------------------------------------------------------- the pages' worked numbers


def test_per_channel_decay_toy(golden):
    """A memory line [10, 10] across the two key channels decays to [9, 2] under a = [0.9, 0.2]."""
    d = golden["per_channel_decay"]
    a = np.array(d["alpha"])
    S0 = np.zeros((1, 1, 2, 2))
    S0[0, 0, :, 0] = d["memory_line_before"]  # one column of S = one value per key channel
    q = np.array([[1.0, 0.0]])
    k = np.array([[0.6, 0.8]])
    v = np.array([[1.0, -1.0]])
    g = np.log(a)[None]
    beta = np.array([0.0])  # no write: the step is the decay alone
    _, Sf = oracle.recurrent(_one_head(q), _one_head(k), _one_head(v), _one_head(g),
                             beta[None, :, None], S0)
    np.testing.assert_allclose(Sf[0, 0, :, 0], d["memory_line_after"], rtol=0, atol=1e-12)


def test_half_life_toy(golden):
    """Half-lives ln(0.5)/ln(a): about 6.6 tokens and 0.43 tokens, a ratio of about 15."""
    d = golden["half_life"]
    a = np.array(d["alpha"])
    T = 12
    q = np.tile(np.eye(2)[None], (T, 1, 1))  # read each key channel of S
    S0 = np.ones((1, 2, 2, 2))  # one (b, h) pair per head below
    outs = []
    for ch in range(2):
        qq = q[:, ch]
        kk = np.tile(np.array([[1.0, 0.0]]), (T, 1))
        vv = np.zeros((T, 2))
        gg = np.tile(np.log(a)[None], (T, 1))
        o, _ = oracle.recurrent(_one_head(qq), _one_head(kk), _one_head(vv), _one_head(gg),
                                np.zeros((1, T, 1)), S0[:, :1])
        outs.append(o[0, :, 0, 0])
    t = np.arange(1, T + 1)
    hl = []
    for ch in range(2):
        # S_t = a^t exactly, so log S_t / t recovers ln a; the half-life is ln 0.5 / ln a
        slope = np.log(outs[ch]) / t
        np.testing.assert_allclose(slope, np.log(a[ch]), rtol=1e-12)
        hl.append(math.log(0.5) / slope.mean())
    for h, printed, dec in zip(hl, d["half_life_tokens_printed"], d["printed_decimals"]):
        assert round(h, dec) == printed
    assert round(hl[0] / hl[1], d["ratio_decimals"]) == d["ratio_printed"]
    # the state really is halved between token 6 and token 7 on the retaining channel
    assert outs[0][5] > 0.5 > outs[0][6]


@pytest.mark.parametrize("prior_scale", [0.0, 1.0, 37.5])
def test_delta_correction_toy(golden, prior_scale):
    """beta = 1 write on channel 2 gives exactly [4, 4] whatever was there; two gate steps of
    0.2 later 4 * 0.2^2 = 0.160; the same write on channel 1 keeps 3.240."""
    d = golden["delta_correction"]
    a = np.array(d["alpha"])
    rng = np.random.default_rng(7)
    for ch, after in ((1, d["channel_2_after_two_steps"]), (0, d["channel_1_after_two_steps"])):
        S0 = prior_scale * rng.standard_normal((1, 1, 2, 2))
        T = 1 + d["gate_steps_after_write"]
        k = np.zeros((T, 2))
        k[0, ch] = 1.0
        v = np.zeros((T, 2))
        v[0] = d["value_written"]
        g = np.tile(np.log(a)[None], (T, 1))
        beta = np.zeros(T)
        beta[0] = d["beta"]
        q = np.zeros((T, 2))
        q[:, ch] = 1.0  # o_t = S_t^T e_ch is row ch of the post-update state
        o, _ = oracle.recurrent(_one_head(q), _one_head(k), _one_head(v), _one_head(g),
                                beta[None, :, None], S0)
        np.testing.assert_allclose(o[0, 0, 0], d["row_after_write_on_channel_2"], atol=1e-12)
        np.testing.assert_allclose(o[0, -1, 0], [after, after], atol=1e-12)


# ---------------------------------------------------------------- closed forms and brute force


def test_alpha_one_is_textbook_delta_rule():
    """g = 0 (alpha = 1) reduces to S_t = (I - beta k k^T) S_{t-1} + beta k v^T."""
    T, dk, dv = 20, 5, 3
    q, k, v, g, beta = _rand_inputs(1, T, 1, dk, dv, RNG)
    g[:] = 0.0
    S0 = RNG.standard_normal((1, 1, dk, dv))
    o, Sf = oracle.recurrent(q, k, v, g, beta, S0)
    S = S0[0, 0].copy()
    for t in range(T):
        kt = k[0, t, 0]
        S = (np.eye(dk) - beta[0, t, 0] * np.outer(kt, kt)) @ S + beta[0, t, 0] * np.outer(kt, v[0, t, 0])
        np.testing.assert_allclose(o[0, t, 0], S.T @ q[0, t, 0], atol=1e-12)
    np.testing.assert_allclose(Sf[0, 0], S, atol=1e-12)


def test_beta_zero_closed_form():
    """beta = 0: S_t = Diag(gamma^{1->t}) S_0 and o_t = S_0^T (gamma^{1->t} * q_t)."""
    T, dk, dv = 17, 6, 4
    q, k, v, g, beta = _rand_inputs(2, T, 3, dk, dv, RNG)
    beta[:] = 0.0
    S0 = RNG.standard_normal((2, 3, dk, dv))
    o, Sf = oracle.recurrent(q, k, v, g, beta, S0)
    gam = np.exp(np.cumsum(g, axis=1))  # [B, T, H, dk], inclusive products of alpha
    for b in range(2):
        for h in range(3):
            for t in range(T):
                np.testing.assert_allclose(o[b, t, h], S0[b, h].T @ (gam[b, t, h] * q[b, t, h]),
                                           atol=1e-12)
            np.testing.assert_allclose(Sf[b, h], gam[b, -1, h][:, None] * S0[b, h], atol=1e-12)


def test_first_token_reads_post_update_state():
    """T = 1, S_0 = 0: S_1 = beta k v^T, so o_1 = beta (k . q) v (not 0)."""
    dk, dv = 7, 5
    q, k, v, g, beta = _rand_inputs(1, 1, 1, dk, dv, RNG)
    o, _ = oracle.recurrent(q, k, v, g, beta)
    expect = beta[0, 0, 0] * (k[0, 0, 0] @ q[0, 0, 0]) * v[0, 0, 0]
    np.testing.assert_allclose(o[0, 0, 0], expect, atol=1e-14)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_bruteforce_products_of_transitions(T):
    """S_T = (M_T...M_1) S_0 + sum_j (M_T...M_{j+1}) beta_j k_j v_j^T with
    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t), expanded explicitly."""
    dk, dv = 4, 3
    q, k, v, g, beta = _rand_inputs(1, T, 1, dk, dv, RNG, unit=False, beta_lo=-0.5, beta_hi=1.5)
    S0 = RNG.standard_normal((1, 1, dk, dv))
    o, Sf = oracle.recurrent(q, k, v, g, beta, S0)
    M = [(np.eye(dk) - beta[0, t, 0] * np.outer(k[0, t, 0], k[0, t, 0])) @ np.diag(np.exp(g[0, t, 0]))
         for t in range(T)]
    for t_end in range(1, T + 1):
        prod = np.eye(dk)
        for t in range(t_end):
            prod = M[t] @ prod
        S = prod @ S0[0, 0]
        for j in range(t_end):
            tail = np.eye(dk)
            for t in range(j + 1, t_end):
                tail = M[t] @ tail
            S = S + tail @ (beta[0, j, 0] * np.outer(k[0, j, 0], v[0, j, 0]))
        np.testing.assert_allclose(o[0, t_end - 1, 0], S.T @ q[0, t_end - 1, 0], atol=1e-12)
        if t_end == T:
            np.testing.assert_allclose(Sf[0, 0], S, atol=1e-12)


def test_transition_is_contraction_invariant():
    """For |k| = 1 and beta in [0, 1], ||M_t||_2 <= 1, so ||S_t||_F <= ||S_{t-1}||_F + beta ||v||."""
    T, dk, dv = 40, 8, 8
    q, k, v, g, beta = _rand_inputs(1, T, 1, dk, dv, RNG)
    S = RNG.standard_normal((1, 1, dk, dv)) * 3.0
    for t in range(T):
        sl = slice(t, t + 1)
        _, Sn = oracle.recurrent(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S)
        bound = np.linalg.norm(S) + beta[0, t, 0] * np.linalg.norm(v[0, t, 0])
        assert np.linalg.norm(Sn) <= bound + 1e-12
        S = Sn


def test_split_resume_equivalence():
    """Running T tokens equals running T1 tokens, then T - T1 from the returned state."""
    T, dk, dv = 33, 6, 5
    q, k, v, g, beta = _rand_inputs(2, T, 2, dk, dv, RNG)
    S0 = RNG.standard_normal((2, 2, dk, dv))
    o, Sf = oracle.recurrent(q, k, v, g, beta, S0)
    for T1 in (0, 1, 16, 32, 33):
        a = slice(0, T1)
        b = slice(T1, T)
        o1, S1 = oracle.recurrent(q[:, a], k[:, a], v[:, a], g[:, a], beta[:, a], S0)
        o2, S2 = oracle.recurrent(q[:, b], k[:, b], v[:, b], g[:, b], beta[:, b], S1)
        np.testing.assert_allclose(np.concatenate([o1, o2], 1), o, atol=1e-12)
        np.testing.assert_allclose(S2, Sf, atol=1e-12)


def test_threads_do_not_change_results():
    q, k, v, g, beta = _rand_inputs(3, 21, 4, 9, 7, RNG)
    a = oracle.recurrent(q, k, v, g, beta, nthreads=1)
    b = oracle.recurrent(q, k, v, g, beta, nthreads=8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- packed batches and decode


def test_varlen_equals_independent_sequences():
    H, dk, dv = 3, 6, 5
    cu = np.array([0, 1, 1, 9, 40, 41], dtype=np.int32)  # includes an empty sequence
    T = int(cu[-1])
    q, k, v, g, beta = _rand_inputs(1, T, H, dk, dv, RNG)
    N = len(cu) - 1
    S0 = RNG.standard_normal((N, H, dk, dv))
    o, Sf = oracle.recurrent_varlen(q, k, v, g, beta, cu, S0)
    for s in range(N):
        sl = slice(int(cu[s]), int(cu[s + 1]))
        oi, Si = oracle.recurrent(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S0[s:s + 1])
        np.testing.assert_array_equal(o[:, sl], oi)
        np.testing.assert_array_equal(Sf[s], Si[0])


def test_varlen_rejects_bad_offsets():
    q, k, v, g, beta = _rand_inputs(1, 10, 1, 2, 2, RNG)
    with pytest.raises(ValueError):
        oracle.recurrent_varlen(q, k, v, g, beta, np.array([0, 5, 3, 10], dtype=np.int32))
    with pytest.raises(ValueError):
        oracle.recurrent_varlen(q, k, v, g, beta, np.array([0, 5, 9], dtype=np.int32))


def test_decode_step_is_one_token():
    N, H, dk, dv = 3, 2, 6, 4
    q, k, v, g, beta = _rand_inputs(N, 1, H, dk, dv, RNG)
    S = RNG.standard_normal((N, H, dk, dv))
    o, Sn = oracle.decode_step(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S)
    o_ref, S_ref = oracle.recurrent(q, k, v, g, beta, S)
    np.testing.assert_array_equal(o, o_ref[:, 0])
    np.testing.assert_array_equal(Sn, S_ref)


# ---------------------------------------------------------------- the block (chunkwise) form


@pytest.mark.parametrize("C", [1, 2, 3, 8, 16, 64])
def test_chunkwise_equals_recurrent(C):
    """The block form is exact: same outputs and final state for every block size, including a
    ragged last block."""
    T, dk, dv = 37, 6, 5
    q, k, v, g, beta = _rand_inputs(1, T, 2, dk, dv, RNG)
    S0 = RNG.standard_normal((1, 2, dk, dv))
    o, Sf = oracle.recurrent(q, k, v, g, beta, S0)
    oc, Sc = cw.chunkwise(q, k, v, g, beta, C, S0)
    np.testing.assert_allclose(oc, o, atol=1e-11, rtol=0)
    np.testing.assert_allclose(Sc, Sf, atol=1e-11, rtol=0)


@pytest.mark.parametrize("C", [64, 128])
def test_chunkwise_equals_recurrent_full_width(C):
    """d_k = d_v = 128 and the page's block sizes, with decays down to g_min = -5."""
    T = C + 19
    q, k, v, g, beta = _rand_inputs(1, T, 1, 128, 128, RNG)
    o, Sf = oracle.recurrent(q, k, v, g, beta)
    oc, Sc = cw.chunkwise(q, k, v, g, beta, C)
    scale = np.abs(o).max()
    np.testing.assert_allclose(oc, o, atol=1e-10 * scale, rtol=0)
    np.testing.assert_allclose(Sc, Sf, atol=1e-10 * max(1.0, np.abs(Sf).max()), rtol=0)


def test_block_transition_matches_product_of_M_t():
    """M_block = Diag(gamma_L) - Khat^T W equals M_L ... M_1, and S' = M S + S~."""
    L, dk, dv = 9, 5, 4
    q, k, v, g, beta = _rand_inputs(1, L, 1, dk, dv, RNG)
    K, V, G, bt = k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0]
    M, S_tilde = cw.block_transition(K, V, G, bt)
    prod = np.eye(dk)
    for t in range(L):
        prod = (np.eye(dk) - bt[t] * np.outer(K[t], K[t])) @ np.diag(np.exp(G[t])) @ prod
    np.testing.assert_allclose(M, prod, atol=1e-12)
    S = RNG.standard_normal((dk, dv))
    _, S_next = cw.block_step(q[0, :, 0], K, V, G, bt, S)
    np.testing.assert_allclose(M @ S + S_tilde, S_next, atol=1e-12)
    _, S_zero = oracle.recurrent(q, k, v, g, beta)
    np.testing.assert_allclose(S_tilde, S_zero[0, 0], atol=1e-12)


def test_segment_composition_is_associative_and_exact():
    """(M_b, S~_b) o (M_a, S~_a) = (M_b M_a, M_b S~_a + S~_b); composing the segments of a
    sequence in any grouping reproduces the recurrent final state (context parallelism)."""
    dk, dv = 6, 4
    q, k, v, g, beta = _rand_inputs(1, 30, 1, dk, dv, RNG)
    cuts = [0, 7, 19, 30]
    pairs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        pairs.append(cw.block_transition(k[0, a:b, 0], v[0, a:b, 0], g[0, a:b, 0], beta[0, a:b, 0]))
    left = cw.compose(pairs[2], cw.compose(pairs[1], pairs[0]))
    right = cw.compose(cw.compose(pairs[2], pairs[1]), pairs[0])
    np.testing.assert_allclose(left[0], right[0], atol=1e-12)
    np.testing.assert_allclose(left[1], right[1], atol=1e-12)
    S0 = RNG.standard_normal((1, 1, dk, dv))
    _, Sf = oracle.recurrent(q, k, v, g, beta, S0)
    np.testing.assert_allclose(left[0] @ S0[0, 0] + left[1], Sf[0, 0], atol=1e-12)


def test_forward_substitution_inverse():
    A = np.tril(RNG.standard_normal((12, 12)), -1) * 0.3
    T = cw.forward_substitution_inverse(A)
    np.testing.assert_allclose(T @ (np.eye(12) + A), np.eye(12), atol=1e-12)
