"""FP64 chunked (WY / UT-transform) restatement of the KDA delta rule.

TEST INFRASTRUCTURE ONLY. It exists to pin the chunk algebra that the CUDA
prefill uses against the sequential oracle (kda_oracle.c): the two must agree
to rounding on every chunk size. It shares nothing with the CUDA library.

The recurrence (kimi_k3.c header, "KDA per-head recurrence"), per token r:
    S_r = (I - b_r k_r k_r^T) Diag(a_r) S_{r-1} + b_r k_r v_r^T,   o_r = S_r^T q_r.
Written with u_r = b_r (v_r - (Diag(a_r) S_{r-1})^T k_r) it is
    S_r = Diag(a_r) S_{r-1} + k_r u_r^T.
Unrolling over a chunk of n tokens that starts from state S0, with the
cumulative log decay G_r = sum_{i<=r} log a_i (a vector over the key dim) and
E(r, i) = exp(G_r - G_i) (elementwise, <= 1 for i <= r):
    A[r, i]  = b_r * sum_c k_r[c] k_i[c] E(r, i)[c]         (i < r; 0 otherwise)
    (I + A) U = Diag(b) V - Diag(b) (K o exp(G)) S0          -> T = (I + A)^-1
    W  = T Diag(b) (K o exp(G)),  U' = T Diag(b) V,  U = U' - W S0
    O  = (Q o exp(G)) S0 + (P o M) U,  P[r, i] = sum_c q_r[c] k_i[c] E(r, i)[c],
         M the inclusive lower-triangular mask (i <= r)
    S_n = Diag(exp(G_n)) S0 + (K o exp(G_n - G))^T U
This is an exact algebraic rewrite; no term is dropped.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def chunk_step(S0: np.ndarray, q, k, v, alpha, beta):
    """One chunk. q,k,v,alpha: [n, d]; beta: [n]. Returns (O [n, d], S_n [d, d])."""
    q, k, v, alpha = (np.asarray(x, dtype=np.float64) for x in (q, k, v, alpha))
    beta = np.asarray(beta, dtype=np.float64)
    n, d = k.shape
    G = np.cumsum(np.log(alpha), axis=0)                      # [n, d]
    E = np.exp(G[:, None, :] - G[None, :, :])                 # E[r, i, c] = exp(G_r - G_i)
    strict = np.tril(np.ones((n, n)), -1)
    incl = np.tril(np.ones((n, n)))
    A = beta[:, None] * np.einsum("rc,ic,ric->ri", k, k, E * strict[:, :, None])
    P = np.einsum("rc,ic,ric->ri", q, k, E * incl[:, :, None])
    L = np.eye(n) + A
    Kg = k * np.exp(G)
    W = solve_triangular(L, beta[:, None] * Kg, lower=True, unit_diagonal=True)
    Up = solve_triangular(L, beta[:, None] * v, lower=True, unit_diagonal=True)
    U = Up - W @ S0
    O = (q * np.exp(G)) @ S0 + (P * incl) @ U
    Sn = np.exp(G[-1])[:, None] * S0 + (k * np.exp(G[-1][None, :] - G)).T @ U
    return O, Sn


def run_chunked(S0: np.ndarray, q, k, v, alpha, beta, C: int):
    """All tokens in chunks of C (the last one ragged). Returns (O [T, d], S_T)."""
    T = len(beta)
    S = np.array(S0, dtype=np.float64, copy=True)
    outs = []
    for s in range(0, T, C):
        e = min(T, s + C)
        O, S = chunk_step(S, q[s:e], k[s:e], v[s:e], alpha[s:e], beta[s:e])
        outs.append(O)
    if not outs:
        return np.zeros((0, S.shape[1])), S
    return np.concatenate(outs, axis=0), S
