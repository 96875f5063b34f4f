"""Chunkwise form of KDA in fp64 (test infrastructure; see oracle/__init__.py).

This is the chunk algebra of 'From Linear Attention to KDA' (blog-3d3.pages.dev/
posts/150), §7.1-7.3, with the per-channel decay of §7.2 folded in. The page leaves
that last fold open ("adding the decay rescaling of the second step gives the full
A and V~ of the paper"); the reading taken here is the plainest one: substitute the
ansatz
    S_i = Diag(g_i) S_0 + sum_{j<=i} Diag(g_i / g_j) k_j u_j^T,   g_i = a_1 * ... * a_i,
into the recurrence S_i = (I - b_i k_i k_i^T) Diag(a_i) S_{i-1} + b_i k_i v_i^T, exactly
as §7.3 does without decay. Matching terms gives, inside one chunk (positions 1..L):

    G_i      = sum_{m<=i} log a_m                       (cumulative log decay, per channel)
    Akk[i,j] = b_i * sum_c k_i[c] k_j[c] exp(G_i[c] - G_j[c])      j < i
    Aqk[i,j] =       sum_c q_i[c] k_j[c] exp(G_i[c] - G_j[c])      j <= i
    (I + Akk) U = B V - B Khat S_0,   Khat_i = k_i * exp(G_i)       (the UT system, §7.3)
    W  = (I + Akk)^-1 B Khat,   U' = (I + Akk)^-1 B V,   U = U' - W S_0
    O  = Qhat S_0 + Aqk U,       Qhat_i = q_i * exp(G_i)
    S_L = Diag(exp(G_L)) S_0 + sum_j Diag(exp(G_L - G_j)) k_j u_j^T

The triangular system is solved with a library routine (scipy's solve_triangular,
unit lower). Decays are formed directly as exp(G_i - G_j) (no factoring), so nothing
overflows in fp64. With delta=False the correction is dropped (Akk = 0, W = 0).

This function exists to pin the chunk algebra (against the recurrence and the
page's worked example in §7.4); the CUDA path is compared with the recurrence.
"""
import numpy as np
from scipy.linalg import solve_triangular


def chunkwise(q, k, v, la, beta, S0, C, delta=True, return_u=False):
    """One sequence, one head. q, k, la: [T, dk]; v: [T, dv]; beta: [T]; S0: [dk, dv].

    Returns (o [T, dv], S_T [dk, dv]) and, if return_u, the list of per-chunk U.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    la = np.asarray(la, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    S = np.array(S0, dtype=np.float64, copy=True)
    T = q.shape[0]
    dv = v.shape[1]
    o = np.zeros((T, dv), dtype=np.float64)
    us = []
    for s in range(0, T, C):
        e = min(s + C, T)
        L = e - s
        Q, K, V, b = q[s:e], k[s:e], v[s:e], beta[s:e]
        G = np.cumsum(la[s:e], axis=0)                       # [L, dk]
        decay = np.exp(G[:, None, :] - G[None, :, :])        # [L, L, dk]: exp(G_i - G_j)
        lower_strict = np.tril(np.ones((L, L)), -1)
        lower = np.tril(np.ones((L, L)), 0)
        Aqk = np.einsum("ic,jc,ijc->ij", Q, K, np.where(lower[:, :, None] > 0, decay, 0.0))
        if delta:
            Akk = b[:, None] * np.einsum("ic,jc,ijc->ij", K, K,
                                         np.where(lower_strict[:, :, None] > 0, decay, 0.0))
        else:
            Akk = np.zeros((L, L))
        M = np.eye(L) + Akk
        Khat = K * np.exp(G)
        Qhat = Q * np.exp(G)
        Uprime = solve_triangular(M, b[:, None] * V, lower=True, unit_diagonal=True)
        if delta:
            W = solve_triangular(M, b[:, None] * Khat, lower=True, unit_diagonal=True)
        else:
            W = np.zeros_like(Khat)
        U = Uprime - W @ S
        o[s:e] = Qhat @ S + Aqk @ U
        Kend = K * np.exp(G[-1][None, :] - G)                # k_j * g_L / g_j
        S = np.exp(G[-1])[:, None] * S + Kend.T @ U
        us.append(U)
    if return_u:
        return o, S, us
    return o, S
