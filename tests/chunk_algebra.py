"""fp64 numpy restatement of the chunk (UT/WY) form of the gated delta rule.

Test helper only: it pins the chunk algebra that the CUDA kernels follow to
the token-by-token oracle, and the oracle never uses it.

Within a chunk of C tokens with start state S0 (V x K), with gamma the
inclusive cumulative sum of g inside the chunk and b = exp(gamma):
  A   = strictly-lower( diag(beta) K K^T * Gamma ),  Gamma_ij = exp(gamma_i - gamma_j)
  T   = (I + A)^-1 diag(beta)
  W   = T diag(b) K,  U = T V            (UT / WY transform)
  U'  = U - W S0^T                        (the corrected writes)
  O   = scale * ( diag(b) Q S0^T + (Q K^T * Gamma * causal) U' )
  S1  = b_last S0 + U'^T diag(exp(gamma_last - gamma)) K
and, split by linearity in S0, S1 = S0 Mc + U^T D K with
  Mc  = b_last I - W^T D K.
"""
import numpy as np


def _gamma_matrix(gam):
    n = len(gam)
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    diff = np.where(i >= j, gam[:, None] - gam[None, :], -np.inf)
    return np.exp(diff)  # zero above the diagonal


def chunked_head(q, k, v, g, beta, S0, scale, C):
    """One sequence, one head.  q, k [T, K]; v [T, V]; g, beta [T]; S0 [V, K]."""
    T = k.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        Kc, Qc, Vc, gc, bc = k[sl], q[sl], v[sl], g[sl], beta[sl]
        n = Kc.shape[0]
        gam = np.cumsum(gc)
        b = np.exp(gam)
        G = _gamma_matrix(gam)
        A = np.tril(bc[:, None] * (Kc @ Kc.T) * G, -1)
        Tm = np.linalg.solve(np.eye(n) + A, np.diag(bc))
        W = Tm @ (b[:, None] * Kc)
        U = Tm @ Vc
        Up = U - W @ S.T
        P = (Qc @ Kc.T) * G
        o[sl] = scale * ((b[:, None] * Qc) @ S.T + P @ Up)
        d = np.exp(gam[-1] - gam)
        S = np.exp(gam[-1]) * S + Up.T @ (d[:, None] * Kc)
    return o, S


def chunk_transition(k, g, beta, C):
    """M of a token range via the per-chunk Mc = b_last I - W^T D K chained."""
    T, K = k.shape
    M = np.eye(K)
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        Kc, gc, bc = k[sl], g[sl], beta[sl]
        n = Kc.shape[0]
        gam = np.cumsum(gc)
        b = np.exp(gam)
        G = _gamma_matrix(gam)
        A = np.tril(bc[:, None] * (Kc @ Kc.T) * G, -1)
        Tm = np.linalg.solve(np.eye(n) + A, np.diag(bc))
        W = Tm @ (b[:, None] * Kc)
        d = np.exp(gam[-1] - gam)
        Mc = np.exp(gam[-1]) * np.eye(K) - W.T @ (d[:, None] * Kc)
        M = M @ Mc
    return M
