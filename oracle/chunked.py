"""Chunked (WY / UT-transform) statement of the gated delta rule, fp64 numpy.

TEST INFRASTRUCTURE ONLY: used by the CPU tests to pin the sequential oracle
(``oracle.forward``) against a second, independently written formulation of
the same method.  It is never called by the product path.

The derivation, for one (sequence, head), in the transposed orientation
H_t = S_t^T (dk x dv), so that the recurrence reads

    H_t = alpha_t (I - beta_t k_t k_t^T) H_{t-1} + beta_t k_t v_t^T,  o_t = H_t^T q_t.

Write u_t = beta_t (v_t - alpha_t H_{t-1}^T k_t); then H_t = alpha_t H_{t-1} + k_t u_t^T.
Inside a chunk of C tokens that starts from the state H0, let G_i be the
inclusive prefix sum of the log-gates g within the chunk, gamma_i = exp(G_i)
and Gamma_ij = exp(G_i - G_j) for i >= j (the unrolled decay weight of
"Model Architecture Walkthrough", section 5.3.1, with a scalar decay).
Unrolling the write inside the chunk gives

    H_i = gamma_i H0 + sum_{j <= i} Gamma_ij k_j u_j^T.

Substituting H_{i-1} into the definition of u_i gives a unit lower-triangular
system for the rows of U (C x dv):

    (I + A) U = diag(beta) V - diag(beta * gamma) K H0,
    A = strictly_lower( diag(beta) K K^T (.) Gamma ),

so U = U~ - W H0 with T = (I + A)^-1, W = T diag(beta * gamma) K and
U~ = T diag(beta) V (the "WY" factors).  The chunk's outputs and the state it
hands to the next chunk are then

    O   = diag(gamma) Q H0 + ( Q K^T (.) Gamma (.) M_incl ) U
    H_C = gamma_C H0 + ( diag(exp(G_C - G)) K )^T U

where M_incl keeps i >= j.  Chunking is in the spirit of the chunk-parallel
algorithm the pages cite ("v1.0 Architecture & Design Spec" section 2.3;
"Optimization Quartet", Triton GDN kernel section 3.2: intra-chunk parallel
work, inter-chunk serial state carry).

Parity status: pinned (tests/test_oracle_pins.py, chunked-vs-sequential).
"""
from __future__ import annotations

import numpy as np


def _unit(q, k, v, g, beta, H0, C):
    L, dk = k.shape
    dv = v.shape[1]
    o = np.zeros((L, dv))
    H = H0.copy()
    for s in range(0, L, C):
        e = min(s + C, L)
        Q, K, V = q[s:e], k[s:e], v[s:e]
        b = beta[s:e]
        G = np.cumsum(g[s:e])
        gam = np.exp(G)
        n = e - s
        ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        lower_incl = ii >= jj
        diff = np.where(lower_incl, G[:, None] - G[None, :], 0.0)
        Gam = np.where(lower_incl, np.exp(diff), 0.0)
        A = np.where(ii > jj, (b[:, None] * (K @ K.T)) * Gam, 0.0)
        Tm = np.linalg.inv(np.eye(n) + A)
        W = Tm @ ((b * gam)[:, None] * K)
        Ut = Tm @ (b[:, None] * V)
        U = Ut - W @ H
        o[s:e] = gam[:, None] * (Q @ H) + ((Q @ K.T) * Gam) @ U
        decay_to_end = np.exp(G[-1] - G)
        H = gam[-1] * H + (decay_to_end[:, None] * K).T @ U
    return o, H


def forward(q, k, v, g, beta, initial_state=None, cu_seqlens=None, chunk_size=64):
    """Chunked fp64 forward with the same shapes and semantics as ``oracle.forward``."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    B, T, H, dk = q.shape
    dv = v.shape[3]
    if cu_seqlens is None:
        seqs = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens, np.int64)
        seqs = [(0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
    N = len(seqs)
    o = np.zeros((B, T, H, dv))
    sN = np.zeros((N, H, dk, dv))
    for n, (b, s, e) in enumerate(seqs):
        for h in range(H):
            H0 = np.zeros((dk, dv)) if initial_state is None else \
                np.asarray(initial_state, np.float64)[n, h]
            on, Hn = _unit(q[b, s:e, h], k[b, s:e, h], v[b, s:e, h],
                           g[b, s:e, h], beta[b, s:e, h], H0, chunk_size)
            o[b, s:e, h] = on
            sN[n, h] = Hn
    return o, sN
