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

chunked_head_bwd takes the same chunk form backward (reverse mode through each
of the steps above, chunk by chunk from the last).  The state gradient runs as
the transposed chain dS0 = dS1 Mc^T + (terms local to the chunk), which is what
a backward scan kernel follows.
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


def chunked_head_bwd(q, k, v, g, beta, S0, scale, C, do, dST):
    """Gradients (dq, dk, dv, dg, dbeta, dS0) of L = <do, o> + <dST, S_T> for chunked_head.

    The chunk start states come from a forward pass; then, from the last chunk to the
    first, each step of the chunk form above is taken back in reverse order:
      S1 = b_last S0 + U'^T D K        O = scale (diag(b) Q S0^T + P U'),  P = (Q K^T) * Gamma
      U' = U - W S0^T                  W = T diag(b) K,  U = T V,  T = (I + A)^-1 diag(beta)
      A = strictly-lower(diag(beta) (K K^T) * Gamma)
    and the gradients of gamma, b = exp(gamma), d = exp(gamma_last - gamma) and Gamma go
    to g through the cumulative sum (dg_i = sum over j >= i of dgamma_j).
    """
    T, K = k.shape
    starts = []
    S = np.array(S0, dtype=np.float64, copy=True)
    for c0 in range(0, T, C):
        starts.append(S.copy())
        sl = slice(c0, min(c0 + C, T))
        S = chunked_head(q[sl], k[sl], v[sl], g[sl], beta[sl], S, scale, C)[1]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros(T), np.zeros(T)
    dS = np.array(dST, dtype=np.float64, copy=True)
    for ci in reversed(range(len(starts))):
        sl = slice(ci * C, min(ci * C + C, T))
        S = starts[ci]
        Kc, Qc, Vc, gc, bc = k[sl], q[sl], v[sl], g[sl], beta[sl]
        n = Kc.shape[0]
        gam = np.cumsum(gc)
        b = np.exp(gam)
        d = np.exp(gam[-1] - gam)
        G = _gamma_matrix(gam)
        KK = Kc @ Kc.T
        A = np.tril(bc[:, None] * KK * G, -1)
        Z = np.linalg.inv(np.eye(n) + A)
        Tm = Z * bc[None, :]
        Kb = b[:, None] * Kc
        W = Tm @ Kb
        U = Tm @ Vc
        Up = U - W @ S.T
        QK = Qc @ Kc.T
        P = QK * G
        Ot = scale * do[sl]
        db = np.zeros(n)
        # S1 = b_last S0 + U'^T D K
        dS0 = b[-1] * dS
        db[-1] += np.sum(S * dS)
        dUp = (d[:, None] * Kc) @ dS.T
        dK = (d[:, None] * Up) @ dS
        dd = np.einsum("iv,vk,ik->i", Up, dS, Kc)
        # O = scale (diag(b) Q S0^T + P U')
        dQ = (b[:, None] * Ot) @ S
        dS0 += Ot.T @ (b[:, None] * Qc)
        db += np.einsum("iv,vk,ik->i", Ot, S, Qc)
        dP = Ot @ Up.T
        dUp += P.T @ Ot
        dQ += (dP * G) @ Kc
        dK += (dP * G).T @ Qc
        dG = dP * QK
        # U' = U - W S0^T
        dW = -dUp @ S
        dS0 -= dUp.T @ W
        # W = T diag(b) K, U = T V
        dT = dW @ Kb.T + dUp @ Vc.T
        dKb = Tm.T @ dW
        dK += b[:, None] * dKb
        db += np.sum(Kc * dKb, axis=1)
        dV = Tm.T @ dUp
        # T = Z diag(beta), Z = (I + A)^-1
        dbt = np.sum(dT * Z, axis=0)
        dA = np.tril(-Z.T @ (dT * bc[None, :]) @ Z.T, -1)
        # A = strictly-lower(diag(beta) (K K^T) * Gamma)
        dbt += np.sum(dA * KK * G, axis=1)
        dKK = bc[:, None] * dA * G
        dG += bc[:, None] * dA * KK
        dK += (dKK + dKK.T) @ Kc
        # gamma through Gamma, b and d, then g through the cumulative sum
        dGG = np.tril(dG * G)
        dgam = dGG.sum(axis=1) - dGG.sum(axis=0) + db * b - dd * d
        dgam[-1] += np.sum(dd * d)
        dq[sl], dk[sl], dv[sl] = dQ, dK, dV
        dg[sl] = np.cumsum(dgam[::-1])[::-1]
        dbeta[sl] = dbt
        dS = dS0
    return dq, dk, dv, dg, dbeta, dS
