"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

None of these retypes the oracle's token loop: each checks a closed form, an
invariant, a special case or a brute-force dense-matrix evaluation of the
printed equations.

Sources: "Tail-Replay: Escaping the Curse of Linear Attention in Prefix
Caching for Hybrid LLMs", section 2 Eq. (1) (the GDN update and alpha in
(0, 1]) and section 3 Eq. (2) (replay from a zero state); "LinearKV: One
Cached State Suffices for Position-Independent Caching in Hybrid LLMs",
composition passage (affine chunk map, exact closed-form composition).
"""
import numpy as np
import pytest

import oracle
from gated_deltanet_state_chunked_gb300 import synthetic


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _unit(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _case(T, h_k, h_v, d_k, d_v, seed, gate_scale=0.1):
    x = synthetic.make_replay_inputs([T], h_k, h_v, d_k, d_v, dtype="f32", seed=seed, gate_scale=gate_scale)
    return x


# ---------------------------------------------------------------- special cases of Eq. (1)

def test_beta_zero_is_pure_decay():
    """beta = 0 leaves only the gate: S_t = alpha_t S_{t-1}, so
    S_T = exp(sum g) S0 and o_t = exp(G_t) S0 q_t."""
    rng = _rng(1)
    T, dk, dv = 9, 6, 5
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0.0, 0.5, size=(T, 1))
    beta = np.zeros((T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk))
    S, O = oracle.replay(q, k, v, g, beta, [0, T], S0, l2norm_qk=False)
    G = np.cumsum(g[:, 0])
    np.testing.assert_allclose(S[0, 0], np.exp(G[-1]) * S0[0, 0], rtol=1e-13, atol=1e-15)
    for t in range(T):
        np.testing.assert_allclose(O[t, 0], np.exp(G[t]) * (S0[0, 0] @ q[t, 0]), rtol=1e-12, atol=1e-14)
    # and with a zero initial state everything stays exactly zero
    S, O = oracle.replay(q, k, v, g, beta, [0, T], None, l2norm_qk=False)
    assert not S.any() and not O.any()


def test_unit_gate_full_beta_projects_key_out():
    """alpha = beta = 1, unit k, v = 0: S_t = S_{t-1}(I - k k^T) removes the k
    direction, so S_t k_t = 0 (read out with q_t = k_t)."""
    rng = _rng(2)
    T, dk, dv = 7, 8, 4
    k = _unit(rng, (T, 1, dk))
    v = np.zeros((T, 1, dv))
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk))
    S, O = oracle.replay(k, k, v, g, beta, [0, T], S0, l2norm_qk=False)
    np.testing.assert_allclose(O, 0.0, atol=1e-13)
    np.testing.assert_allclose(S[0, 0] @ k[-1, 0], 0.0, atol=1e-13)


def test_delta_rule_write_reads_back_value():
    """alpha = beta = 1, unit k: S_t k_t = S_{t-1}(k_t - k_t) + v_t = v_t, so
    the readout with q_t = k_t returns v_t exactly (the delta-rule write)."""
    rng = _rng(3)
    T, dk, dv = 11, 8, 6
    k = _unit(rng, (T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dv, dk))
    S, O = oracle.replay(k, k, v, np.zeros((T, 1)), np.ones((T, 1)), [0, T], S0, l2norm_qk=False)
    np.testing.assert_allclose(O[:, 0], v[:, 0], rtol=1e-12, atol=1e-12)


def test_single_step_action_on_key_and_complement():
    """One step, general alpha and beta, unit k:
    S_1 k = alpha (1 - beta) S0 k + beta v, and S_1 u = alpha S0 u for u orthogonal to k."""
    rng = _rng(4)
    dk, dv = 10, 7
    k = _unit(rng, (1, 1, dk))
    v = rng.standard_normal((1, 1, dv))
    g = np.array([[-0.37]])
    beta = np.array([[0.61]])
    S0 = rng.standard_normal((1, 1, dv, dk))
    S, _ = oracle.replay(k, k, v, g, beta, [0, 1], S0, l2norm_qk=False, want_O=False)
    a, b = np.exp(g[0, 0]), beta[0, 0]
    kk = k[0, 0]
    np.testing.assert_allclose(S[0, 0] @ kk, a * (1 - b) * (S0[0, 0] @ kk) + b * v[0, 0], rtol=1e-12)
    u = rng.standard_normal(dk)
    u -= (u @ kk) * kk
    np.testing.assert_allclose(S[0, 0] @ u, a * (S0[0, 0] @ u), rtol=1e-12, atol=1e-13)


def test_orthonormal_keys_give_outer_product_memory():
    """Orthonormal keys, alpha = beta = 1, S0 = 0: S_T = sum_t v_t k_t^T (a plain
    outer-product associative memory) and S_T k_j = v_j for every j."""
    rng = _rng(5)
    T, dk, dv = 10, 16, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :T].T.reshape(T, 1, dk)
    v = rng.standard_normal((T, 1, dv))
    S, _ = oracle.replay(k, k, v, np.zeros((T, 1)), np.ones((T, 1)), [0, T], l2norm_qk=False, want_O=False)
    expect = sum(np.outer(v[t, 0], k[t, 0]) for t in range(T))
    np.testing.assert_allclose(S[0, 0], expect, rtol=1e-12, atol=1e-13)
    for j in range(T):
        np.testing.assert_allclose(S[0, 0] @ k[j, 0], v[j, 0], rtol=1e-12, atol=1e-13)


def test_scalar_case_closed_form():
    """d_k = d_v = 1: s_t = alpha_t (1 - beta_t k_t^2) s_{t-1} + beta_t v_t k_t, a
    first-order linear recurrence with the solution
    s_T = prod_t a_t * s_0 + sum_t b_t prod_{u>t} a_u."""
    rng = _rng(6)
    T = 40
    k = rng.standard_normal((T, 1, 1))
    q = rng.standard_normal((T, 1, 1))
    v = rng.standard_normal((T, 1, 1))
    g = -rng.uniform(0, 0.3, size=(T, 1))
    beta = rng.uniform(0, 1, size=(T, 1))
    s0 = 0.7
    S, O = oracle.replay(q, k, v, g, beta, [0, T], np.full((1, 1, 1, 1), s0), l2norm_qk=False)
    a = np.exp(g[:, 0]) * (1 - beta[:, 0] * k[:, 0, 0] ** 2)
    b = beta[:, 0] * v[:, 0, 0] * k[:, 0, 0]
    for t in range(T):
        st = np.prod(a[: t + 1]) * s0 + sum(b[j] * np.prod(a[j + 1: t + 1]) for j in range(t + 1))
        assert O[t, 0, 0] == pytest.approx(st * q[t, 0, 0], rel=1e-11, abs=1e-14)
    assert S[0, 0, 0, 0] == pytest.approx(np.prod(a) * s0 + sum(b[j] * np.prod(a[j + 1:]) for j in range(T)), rel=1e-11)


# ---------------------------------------------------------------- brute force with dense matrices

def _dense_left_form(q, k, v, g, beta, X0, scale=1.0):
    """Eq. (1) exactly as printed, on X = S^T (d_k x d_v): X_i = T_i X_{i-1} + beta_i k_i v_i^T
    with T_i = alpha_i (I - beta_i k_i k_i^T) formed as a dense matrix; o_i = X_i^T q_i."""
    T, dk = k.shape
    X = X0.copy()
    outs = []
    for i in range(T):
        Ti = np.exp(g[i]) * (np.eye(dk) - beta[i] * np.outer(k[i], k[i]))
        X = Ti @ X + beta[i] * np.outer(k[i], v[i])
        outs.append(X.T @ (scale * q[i]))
    return X, np.array(outs)


@pytest.mark.parametrize("dk,dv,T", [(5, 3, 7), (4, 6, 12), (1, 1, 5)])
def test_brute_force_dense_transitions(dk, dv, T):
    rng = _rng(7 + dk)
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0, 0.4, size=(T, 1))
    beta = rng.uniform(0, 1, size=(T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk))
    S, O = oracle.replay(q, k, v, g, beta, [0, T], S0, l2norm_qk=False, scale=0.5)
    X, outs = _dense_left_form(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0, 0].T, scale=0.5)
    np.testing.assert_allclose(S[0, 0], X.T, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(O[:, 0], outs, rtol=1e-12, atol=1e-13)


def test_l2norm_flag_is_scale_invariant():
    """With the q/k normalisation flag on, rescaling q and k by positive factors
    changes nothing (up to the 1e-6 epsilon), and unit inputs reproduce the
    unnormalised run."""
    rng = _rng(8)
    T, dk, dv = 20, 8, 8
    q = _unit(rng, (T, 1, dk))
    k = _unit(rng, (T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0, 0.3, size=(T, 1))
    beta = rng.uniform(0, 1, size=(T, 1))
    S_ref, O_ref = oracle.replay(q, k, v, g, beta, [0, T], l2norm_qk=False)
    cq = rng.uniform(2, 5, size=(T, 1, 1))
    ck = rng.uniform(2, 5, size=(T, 1, 1))
    S, O = oracle.replay(q * cq, k * ck, v, g, beta, [0, T], l2norm_qk=True)
    assert oracle.rel_err(S, S_ref) < 1e-7
    assert oracle.rel_err(O, O_ref) < 1e-7


def test_gqa_consecutive_v_heads_share_a_key_head():
    """h_v = 2 h_k: v-heads 2j and 2j+1 read q/k head j (reading of the grouped layout)."""
    x = _case(30, 2, 4, 8, 8, seed=9)
    S, O = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)
    qr = np.repeat(x.q, 2, axis=1)
    kr = np.repeat(x.k, 2, axis=1)
    S2, O2 = oracle.replay(qr, kr, x.v, x.g, x.beta, x.cu_seqlens)
    np.testing.assert_array_equal(S, S2)
    np.testing.assert_array_equal(O, O2)


def test_packed_sequences_are_independent_and_empty_ones_are_identity():
    x = synthetic.make_replay_inputs([13, 0, 29, 1], 1, 2, 8, 4, dtype="f32", seed=10, with_S0=True)
    S, O = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.S0)
    cu = x.cu_seqlens
    for s in range(4):
        a, b = cu[s], cu[s + 1]
        Ss, Os = oracle.replay(x.q[a:b], x.k[a:b], x.v[a:b], x.g[a:b], x.beta[a:b], [0, b - a], x.S0[s:s + 1])
        np.testing.assert_array_equal(S[s], Ss[0])
        np.testing.assert_array_equal(O[a:b], Os)
    np.testing.assert_array_equal(S[1], x.S0[1])  # empty tail: the state is untouched


def test_selected_pairs_match_full_run():
    x = synthetic.make_replay_inputs([17, 23], 2, 4, 8, 8, dtype="f32", seed=11)
    S, O = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)
    sel = [(1, 3), (0, 0)]
    S2, O2 = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, sel=sel)
    for s, h in sel:
        np.testing.assert_array_equal(S2[s, h], S[s, h])
        a, b = x.cu_seqlens[s], x.cu_seqlens[s + 1]
        np.testing.assert_array_equal(O2[a:b, h], O[a:b, h])


# ---------------------------------------------------------------- chunk operator and composition

def test_chunk_operator_equals_dense_product():
    """T_C is the product of the chunk's dense per-token transitions, latest on
    the left; S_local is the state reached from an empty start."""
    rng = _rng(12)
    T, dk, dv = 9, 5, 3
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0, 0.4, size=(T, 1))
    beta = rng.uniform(0, 1, size=(T, 1))
    Tc, Sl = oracle.chunk_operator(k, g, beta, v, [0, T], l2norm_qk=False)
    P = np.eye(dk)
    for i in range(T):
        P = (np.exp(g[i, 0]) * (np.eye(dk) - beta[i, 0] * np.outer(k[i, 0], k[i, 0]))) @ P
    np.testing.assert_allclose(Tc[0, 0], P, rtol=1e-12, atol=1e-14)
    X, _ = _dense_left_form(k[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], np.zeros((dk, dv)))
    np.testing.assert_allclose(Sl[0, 0], X.T, rtol=1e-12, atol=1e-14)


def test_chunk_map_is_affine_in_entering_state():
    """The recurrence is linear in the state, so a chunk maps S_in to
    S_in T_C^T + S_local (pages' form T_C S_in + S_local on the transposed state)."""
    x = synthetic.make_replay_inputs([50], 2, 4, 8, 6, dtype="f32", seed=13, gate_scale=1e-2, with_S0=True)
    S, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.S0, want_O=False)
    Tc, Sl = oracle.chunk_operator(x.k, x.g, x.beta, x.v, x.cu_seqlens)
    pred = np.einsum("hij,hkj->hik", x.S0[0].astype(np.float64), Tc[0]) + Sl[0]
    np.testing.assert_allclose(S[0], pred, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("with_S_in", [False, True])
def test_composition_of_chunk_operators_equals_sequential_replay(with_S_in):
    """Composing the isolated chunks' operators is exact (no approximation of its
    own): compose(chunk ops) == replay of the concatenated tokens."""
    pieces = [37, 64, 5, 50]
    x = synthetic.make_replay_inputs([sum(pieces)], 2, 4, 8, 6, dtype="f32", seed=14, gate_scale=1e-2,
                                     with_S0=with_S_in)
    cu = np.concatenate([[0], np.cumsum(pieces)])
    Tc, Sl = oracle.chunk_operator(x.k, x.g, x.beta, x.v, cu)
    S_in = x.S0[0] if with_S_in else None
    SK = oracle.compose(Tc, Sl, S_in)
    S, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.S0, want_O=False)
    np.testing.assert_allclose(SK, S[0], rtol=1e-11, atol=1e-12)


def test_compose_matches_horner_on_random_operators():
    """On arbitrary matrices the closed form equals chunk-by-chunk application
    S <- S T_j^T + S_local_j (the affine maps applied back to back)."""
    rng = _rng(15)
    K, h, dk, dv = 5, 3, 6, 4
    T = rng.standard_normal((K, h, dk, dk)) * 0.5
    Sl = rng.standard_normal((K, h, dv, dk))
    S_in = rng.standard_normal((h, dv, dk))
    out = oracle.compose(T, Sl, S_in)
    S = S_in.copy()
    for j in range(K):
        S = np.einsum("hij,hkj->hik", S, T[j]) + Sl[j]
    np.testing.assert_allclose(out, S, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.compose(T[:0], Sl[:0], S_in), S_in)
    # without an entering state the result drops S_in carried through every transition
    carried = S_in.copy()
    for j in range(K):
        carried = np.einsum("hij,hkj->hik", carried, T[j])
    np.testing.assert_allclose(oracle.compose(T, Sl, None), S - carried, rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------- replay vs full prefix

def test_replay_error_is_the_carried_prefix_state():
    """Linearity gives S_full - S_replay = S_{L-r} P_tail with P_tail the tail's
    transition product; and since ||I - beta k k^T|| <= 1 for beta in [0, 1] and
    unit k, ||S_full - S_replay|| <= exp(sum_tail g) ||S_{L-r}||."""
    L, r = 120, 40
    x = synthetic.make_replay_inputs([L], 1, 2, 8, 8, dtype="f32", seed=16, gate_scale=2e-2)
    S_full, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, want_O=False)
    a = L - r
    S_rep, _ = oracle.replay(x.q[a:], x.k[a:], x.v[a:], x.g[a:], x.beta[a:], [0, r], want_O=False)
    S_pre, _ = oracle.replay(x.q[:a], x.k[:a], x.v[:a], x.g[:a], x.beta[:a], [0, a], want_O=False)
    Tc, _ = oracle.chunk_operator(x.k[a:], x.g[a:], x.beta[a:], x.v[a:], [0, r])
    diff = S_full[0] - S_rep[0]
    pred = np.einsum("hij,hkj->hik", S_pre[0], Tc[0])
    np.testing.assert_allclose(diff, pred, rtol=1e-10, atol=1e-13)
    for h in range(2):
        bound = np.exp(x.g[a:, h].astype(np.float64).sum()) * np.linalg.norm(S_pre[0, h])
        assert np.linalg.norm(diff[h]) <= bound * (1 + 1e-12)
        assert np.linalg.norm(diff[h]) > 0


def test_output_scale_is_linear():
    x = _case(25, 1, 1, 8, 8, seed=17)
    _, O1 = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, scale=1.0)
    _, O2 = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, scale=0.125)
    np.testing.assert_allclose(O2, 0.125 * O1, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- the parity metric itself

def test_rel_err_on_hand_computed_vectors():
    """oracle.rel_err is the one comparison every GPU parity test makes, so it is pinned to
    values worked out by hand: ||x - ref|| / ||ref|| over the whole tensor, falling back to the
    absolute norm when ref is zero."""
    assert oracle.rel_err([3.0, 4.0], [0.0, 0.0]) == 5.0          # zero reference: absolute norm
    assert oracle.rel_err([1.0, 1.0], [1.0, 0.0]) == 1.0          # |(0,1)| / |(1,0)|
    assert oracle.rel_err([1.0, 0.0], [1.0, 1.0]) == pytest.approx(2 ** -0.5, rel=1e-15)  # not symmetric
    # a 2x2 tensor: sqrt(1 + 4) / sqrt(9 + 16) over all elements, not row by row
    assert oracle.rel_err([[1.0, 2.0], [3.0, 4.0]], [[0.0, 0.0], [3.0, 4.0]]) == pytest.approx(5 ** 0.5 / 5, rel=1e-15)
    x = np.arange(1.0, 7.0).reshape(2, 3)
    assert oracle.rel_err(x, x) == 0.0
    assert oracle.rel_err(3.0 * x, 3.0 * x) == 0.0
    # one changed element among a thousand is seen, with the value the definition gives
    ref = np.ones(1000)
    y = ref.copy()
    y[517] += 1e-3
    assert oracle.rel_err(y, ref) == pytest.approx(1e-3 / 1000 ** 0.5, rel=1e-9)
    assert oracle.rel_err(y, ref) > 0.0
    # scale invariance: scaling x and ref together leaves it unchanged
    assert oracle.rel_err(7.0 * y, 7.0 * ref) == pytest.approx(oracle.rel_err(y, ref), rel=1e-12)
    # float32 inputs are compared in fp64 (the difference is not rounded away)
    a32 = np.float32(1.0) + np.float32(2 ** -20)
    assert oracle.rel_err(np.array([a32], np.float32), np.array([1.0], np.float32)) == 2 ** -20


# ---------------------------------------------------------------- the scalar-decay (Mamba-2) family

def test_scalar_decay_closed_form():
    """The LinearKV page's other recurrence family has a scalar per-token transition, so the
    state is a decayed sum: S_T = (prod alpha) S0 + sum_t (prod_{s>t} alpha_s) beta_t v_t k_t^T,
    and o_t = S_t q_t reads the state right after token t."""
    rng = _rng(70)
    T, dk, dv = 11, 5, 4
    q, k = rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0.0, 0.6, size=(T, 1))
    beta = rng.uniform(0.1, 1.0, size=(T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk))
    S, O = oracle.replay(q, k, v, g, beta, [0, T], S0, l2norm_qk=False, scalar_decay=True)
    G = np.cumsum(g[:, 0])
    for t in range(T):
        St = np.exp(G[t]) * S0[0, 0]
        for s in range(t + 1):
            St = St + np.exp(G[t] - G[s]) * beta[s, 0] * np.outer(v[s, 0], k[s, 0])
        np.testing.assert_allclose(O[t, 0], St @ q[t, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S[0, 0], St, rtol=1e-12, atol=1e-12)


def test_scalar_decay_brute_force_and_difference_from_gdn():
    """Dense left-form product with T_t = alpha_t I on the transposed state matches; and the same
    inputs under GDN differ exactly by the projection term (a scalar model keeps the k direction
    of the old state, GDN's delta rule removes it)."""
    rng = _rng(71)
    T, dk, dv = 6, 4, 3
    q, k = rng.standard_normal((T, 1, dk)), _unit(rng, (T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0.0, 0.3, size=(T, 1))
    beta = rng.uniform(0.2, 0.9, size=(T, 1))
    S, _ = oracle.replay(q, k, v, g, beta, [0, T], None, l2norm_qk=False, scalar_decay=True)
    St = np.zeros((dk, dv))  # the pages' left form acts on S^T
    for t in range(T):
        Tt = np.exp(g[t, 0]) * np.eye(dk)
        St = Tt @ St + beta[t, 0] * np.outer(k[t, 0], v[t, 0])
    np.testing.assert_allclose(S[0, 0], St.T, rtol=1e-12, atol=1e-12)
    # one token on a known state: scalar keeps S0 k, GDN subtracts beta (S0 k) k^T
    S0 = rng.standard_normal((1, 1, dv, dk))
    a = np.exp(g[:1])
    Ss, _ = oracle.replay(q[:1], k[:1], v[:1], g[:1], beta[:1], [0, 1], S0, l2norm_qk=False, scalar_decay=True)
    Sg, _ = oracle.replay(q[:1], k[:1], v[:1], g[:1], beta[:1], [0, 1], S0, l2norm_qk=False)
    proj = a[0, 0] * beta[0, 0] * np.outer(S0[0, 0] @ k[0, 0], k[0, 0])
    np.testing.assert_allclose(Ss[0, 0] - Sg[0, 0], proj, rtol=1e-12, atol=1e-12)


def test_scalar_decay_chunk_transition_is_a_scalar_and_composition_is_exact():
    """T_C = (prod alpha) I for the scalar family, and composing isolated chunks' operators
    equals the sequential replay of all their tokens."""
    x = synthetic.make_replay_inputs([7, 5, 9], 1, 2, 6, 4, dtype="f32", seed=72, gate_scale=0.5)
    Tc, Sl = oracle.chunk_operator(x.k, x.g, x.beta, x.v, x.cu_seqlens, scalar_decay=True)
    cu = x.cu_seqlens
    for c in range(3):
        for h in range(2):
            prod = np.exp(np.sum(x.g[cu[c]:cu[c + 1], h].astype(np.float64)))
            np.testing.assert_allclose(Tc[c, h], prod * np.eye(6), rtol=1e-13, atol=1e-15)
    S_comp = oracle.compose(Tc, Sl)
    S_seq, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, [0, int(cu[-1])], want_O=False, scalar_decay=True)
    np.testing.assert_allclose(S_comp, S_seq[0], rtol=1e-12, atol=1e-13)
