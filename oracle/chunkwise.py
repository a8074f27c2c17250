"""Chunkwise (block) form of KDA in fp64 NumPy -- TEST INFRASTRUCTURE ONLY.

The pages state that the block form is exact (Kimi K3 wiki, "Glossaire", entry "Chunkwise";
spawnkit course session 17, section 4 "Exécution chunkwise") and that a UT transform turns the
chain of delta projections inside a block into plain matrix products (Glossaire, entry "UT"),
but they print no block equations. The equations below are derived here from the recurrence
(Notations mathématiques, table "Attention et KDA": M_t, S_t, o_t) and are pinned against the
token-by-token oracle by the test-suite; the CUDA kernels implement the same algebra in their
own code.

Derivation, for one block with local positions r = 1..L and incoming state S:
  Gamma_r = sum_{s<=r} g_s (inclusive, per key channel), gamma_r = exp(Gamma_r).
  Writing the update as S_r = Diag(alpha_r) S_{r-1} + k_r u_r^T with
  u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r) and unrolling inside the block gives
     (I + A) U = Diag(beta) V - Diag(beta) (K*gamma) S,
     A_rj = beta_r sum_c k_rc k_jc exp(Gamma_rc - Gamma_jc)         for j < r (strictly lower)
  so with T = (I + A)^{-1} (forward substitution; unit lower triangular):
     W = T Diag(beta) (K*gamma),   U~ = T Diag(beta) V,   U = U~ - W S          (UT transform)
     P_rj = sum_c q_rc k_jc exp(Gamma_rc - Gamma_jc)   for j <= r (Tril keeps the diagonal)
     O    = (Q*gamma) S + P U
     S'   = Diag(gamma_L) S + Khat^T U,   Khat_j = k_j * exp(Gamma_L - Gamma_j)
  and the block transition is M = Diag(gamma_L) - Khat^T W, with S~ = Khat^T U~ the state the
  block reaches from S = 0, so S' = M S + S~ (Notations: M_t and S~; Glossaire: KCP).
"""
from __future__ import annotations

import numpy as np


def forward_substitution_inverse(A: np.ndarray) -> np.ndarray:
    """T = (I + A)^{-1} for strictly lower-triangular A, one row at a time."""
    L = A.shape[0]
    T = np.zeros((L, L))
    for r in range(L):
        row = np.zeros(L)
        row[r] = 1.0
        for j in range(r):
            row -= A[r, j] * T[j]
        T[r] = row
    return T


def block_quantities(Q, K, V, G, beta):
    """All state-independent matrices of one block (shapes [L, d])."""
    Q, K, V, G, beta = (np.asarray(x, dtype=np.float64) for x in (Q, K, V, G, beta))
    L = K.shape[0]
    Gam = np.cumsum(G, axis=0)
    # exp(Gamma_r - Gamma_j) for j <= r only (the exponent is <= 0 there); zero elsewhere
    D = Gam[:, None, :] - Gam[None, :, :]
    lower_incl = np.tril(np.ones((L, L), dtype=bool))
    E = np.where(lower_incl[:, :, None], np.exp(np.where(lower_incl[:, :, None], D, 0.0)), 0.0)
    strict = np.tril(np.ones((L, L)), -1)
    A = beta[:, None] * np.einsum("rc,jc,rjc->rj", K, K, E) * strict
    P = np.einsum("rc,jc,rjc->rj", Q, K, E) * lower_incl
    T = forward_substitution_inverse(A)
    gam = np.exp(Gam)
    W = T @ (beta[:, None] * K * gam)
    Ut = T @ (beta[:, None] * V)
    Khat = K * np.exp(Gam[-1][None, :] - Gam)
    return dict(Gamma=Gam, A=A, T=T, W=W, Ut=Ut, P=P, Khat=Khat, Qg=Q * gam, gamma_L=gam[-1])


def block_step(Q, K, V, G, beta, S):
    """One block: returns (O [L, d_v], S_next)."""
    m = block_quantities(Q, K, V, G, beta)
    U = m["Ut"] - m["W"] @ S
    O = m["Qg"] @ S + m["P"] @ U
    S_next = m["gamma_L"][:, None] * S + m["Khat"].T @ U
    return O, S_next


def block_transition(K, V, G, beta):
    """(M, S~) of one block: S' = M S + S~ for any incoming S."""
    m = block_quantities(np.zeros_like(K), K, V, G, beta)
    M = np.diag(m["gamma_L"]) - m["Khat"].T @ m["W"]
    S_tilde = m["Khat"].T @ m["Ut"]
    return M, S_tilde


def compose(later, earlier):
    """Associative composition of (M, S~) pairs: apply `earlier`, then `later`."""
    Mb, Sb = later
    Ma, Sa = earlier
    return Mb @ Ma, Mb @ Sa + Sb


def chunkwise(q, k, v, g, beta, C: int, S0=None):
    """Block form over a dense batch, same shapes and results as ``oracle.recurrent``."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, T, H, dv))
    Sf = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for n0 in range(0, T, C):
                sl = slice(n0, min(n0 + C, T))
                O, S = block_step(q[b, sl, h], k[b, sl, h], v[b, sl, h], g[b, sl, h],
                                  beta[b, sl, h], S)
                out[b, sl, h] = O
            Sf[b, h] = S
    return out, Sf
