"""The chunk-level regroupings the tensor-core kernels are built on, checked on CPU in fp64
against the oracle's token-by-token recurrence (Tail-Replay section 2 Eq. (1)).

Per chunk of C tokens with normalised keys K (rows k_t), values V, gates G_t (inclusive sums of
g = log alpha inside the chunk, gamma_t = exp(G_t)) and beta:
  A_ts = beta_t exp(G_t - G_s) k_t.k_s (s < t),  M = (I + A)^{-1}
  U~ = M diag(beta) V,  W = M diag(beta gamma) K,  sc_t = exp(G_C - G_t)
  the WY step:       S^T <- gamma_C S^T + K^T diag(sc) (U~ - W S^T)
  the operator step: S^T <- gamma_C S^T + B^T + A^T S^T,
                     A^T = K^T Z K with Z = -diag(sc) M diag(beta gamma),  B^T = K^T diag(sc) U~.
the chunk operator (T_C, S_local) as the WY step on the state augmented with d_k rows,
seeded [0; I], and the scalar-decay family's chunk step (A = 0, M = I, W = 0).  Tokens past a sequence's end inside its last chunk take beta = g = 0 (identity
steps).  The chunk size is small here so that several chunks and a ragged tail fit a small
problem.
"""
import numpy as np
import pytest

import oracle


def _inputs(T, d_k, d_v, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    k = rng.standard_normal((T, d_k))
    v = rng.standard_normal((T, d_v))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    g = -np.log1p(np.exp(rng.standard_normal(T) + 2.0)) * 0.1
    S0 = rng.standard_normal((d_v, d_k))
    return k, v, g, beta, S0


def _chunk_pieces(Kc, Vc, gc, bc):
    C = Kc.shape[0]
    G = np.cumsum(gc)
    gam = np.exp(G)
    A = np.zeros((C, C))
    for t in range(C):
        for s in range(t):
            A[t, s] = bc[t] * np.exp(G[t] - G[s]) * Kc[t] @ Kc[s]
    M = np.linalg.inv(np.eye(C) + A)
    Ut = M @ np.diag(bc) @ Vc
    W = M @ np.diag(bc * gam) @ Kc
    sc = np.exp(G[-1] - G)
    return gam[-1], M, Ut, W, sc, gam


def _run_chunks(k, v, g, beta, S0, C, form):
    T = k.shape[0]
    K = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
    St = S0.T.copy()  # S^T, d_k x d_v
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        Kc = np.zeros((C, K.shape[1])); Kc[:n] = K[c0:c0 + n]
        Vc = np.zeros((C, v.shape[1])); Vc[:n] = v[c0:c0 + n]
        gc = np.zeros(C); gc[:n] = g[c0:c0 + n]
        bc = np.zeros(C); bc[:n] = beta[c0:c0 + n]
        gC, M, Ut, W, sc, gam = _chunk_pieces(Kc, Vc, gc, bc)
        if form == "wy":
            St = gC * St + Kc.T @ np.diag(sc) @ (Ut - W @ St)
        else:
            Z = -np.diag(sc) @ M @ np.diag(bc * gam)
            At = Kc.T @ Z @ Kc
            Bt = Kc.T @ np.diag(sc) @ Ut
            St = gC * St + Bt + At @ St
    return St.T


def _oracle_state(k, v, g, beta, S0):
    T, d_k = k.shape
    d_v = v.shape[1]
    q = np.zeros((T, 1, d_k))
    S, _ = oracle.replay(q, k[:, None, :], v[:, None, :], g[:, None], beta[:, None], np.array([0, T]),
                         S0[None, None], want_O=False)
    return S[0, 0]


@pytest.mark.parametrize("form", ["wy", "operator"])
@pytest.mark.parametrize("T,C", [(37, 8), (64, 16), (5, 8)])
def test_chunk_form_equals_the_token_recurrence(form, T, C):
    k, v, g, beta, S0 = _inputs(T, 6, 5, seed=17 + T + C)
    S_ref = _oracle_state(k, v, g, beta, S0)
    S = _run_chunks(k, v, g, beta, S0, C, form)
    assert oracle.rel_err(S, S_ref) < 1e-12


def test_operator_form_sign_matters():
    """Z with the wrong sign (a plausible slip in the regrouping) is far from the recurrence."""
    k, v, g, beta, S0 = _inputs(40, 6, 5, seed=99)
    S_ref = _oracle_state(k, v, g, beta, S0)
    K = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
    C = 8
    St = S0.T.copy()
    for c0 in range(0, 40, C):
        gC, M, Ut, W, sc, gam = _chunk_pieces(K[c0:c0 + C], v[c0:c0 + C], g[c0:c0 + C], beta[c0:c0 + C])
        Z = +np.diag(sc) @ M @ np.diag(beta[c0:c0 + C] * gam)  # wrong sign
        St = gC * St + K[c0:c0 + C].T @ np.diag(sc) @ Ut + K[c0:c0 + C].T @ Z @ K[c0:c0 + C] @ St
    assert oracle.rel_err(St.T, S_ref) > 1e-3


@pytest.mark.parametrize("T,C", [(29, 8), (48, 16)])
def test_augmented_state_gives_the_chunk_operator(T, C):
    """The chunk operator as the tensor-core kernel builds it: the same WY step run on the state
    augmented with d_k rows P, seeded [S; P] = [0; I] and with no value input for the P rows,
    ends at [S_local; P] where P is the product of the sequence's transitions (stored transposed:
    composition applies S <- S T^T + S_local)."""
    d_k, d_v = 6, 5
    k, v, g, beta, S0 = _inputs(T, d_k, d_v, seed=41 + T)
    K = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
    St = np.zeros((d_k, d_v + d_k))
    St[:, d_v:] = np.eye(d_k)
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        Kc = np.zeros((C, d_k)); Kc[:n] = K[c0:c0 + n]
        Vc = np.zeros((C, d_v + d_k)); Vc[:n, :d_v] = v[c0:c0 + n]
        gc = np.zeros(C); gc[:n] = g[c0:c0 + n]
        bc = np.zeros(C); bc[:n] = beta[c0:c0 + n]
        gC, M, Ut, W, sc, gam = _chunk_pieces(Kc, Vc, gc, bc)
        St = gC * St + Kc.T @ np.diag(sc) @ (Ut - W @ St)
    S_local, P = St.T[:d_v], St.T[d_v:]
    T_ref, Sl_ref = oracle.chunk_operator(k[:, None, :], g[:, None], beta[:, None], v[:, None, :], np.array([0, T]))
    assert oracle.rel_err(S_local, Sl_ref[0, 0]) < 1e-12
    assert oracle.rel_err(P.T, T_ref[0, 0]) < 1e-12
    assert oracle.rel_err(S0 @ P + S_local, _oracle_state(k, v, g, beta, S0)) < 1e-12


@pytest.mark.parametrize("T,C", [(37, 8), (16, 16)])
def test_scalar_decay_chunk_form(T, C):
    """The scalar-transition (Mamba-2) family as the kernels run it: A = 0, M = I and W = 0, so
    the chunk step is S^T <- gamma_C S^T + K^T diag(sc) diag(beta) V (and the operator A^T = 0)."""
    d_k, d_v = 6, 5
    k, v, g, beta, S0 = _inputs(T, d_k, d_v, seed=61 + T)
    K = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
    St = S0.T.copy()
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        Kc = np.zeros((C, d_k)); Kc[:n] = K[c0:c0 + n]
        Vc = np.zeros((C, d_v)); Vc[:n] = v[c0:c0 + n]
        gc = np.zeros(C); gc[:n] = g[c0:c0 + n]
        bc = np.zeros(C); bc[:n] = beta[c0:c0 + n]
        G = np.cumsum(gc)
        sc = np.exp(G[-1] - G)
        St = np.exp(G[-1]) * St + Kc.T @ np.diag(sc * bc) @ Vc
    q = np.zeros((T, 1, d_k))
    S_ref, _ = oracle.replay(q, k[:, None, :], v[:, None, :], g[:, None], beta[:, None], np.array([0, T]),
                             S0[None, None], want_O=False, scalar_decay=True)
    assert oracle.rel_err(St.T, S_ref[0, 0]) < 1e-12
