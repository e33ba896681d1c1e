"""Chunked statement of the backward pass of the gated delta rule, fp64 numpy.

TEST INFRASTRUCTURE ONLY: the CPU tests pin it against the autograd oracle
(``oracle.grad.backward``), so that the chunked algebra of the backward --
the reverse of the WY form in ``oracle.chunked`` -- is checked on its own,
in exact arithmetic up to fp64 rounding.  It is never called by the product
path and shares no code with it.

Per chunk of C = 64 tokens (zero-padded at the end of a sequence: padded
tokens have k = q = v = 0, beta = 0, g = 0 and leave everything unchanged),
with H the state entering the chunk, G the chunk-local prefix sum of g,
gamma = exp(G), Gamma_ij = exp(G_i - G_j), dec_i = exp(G_C - G_i) and, as in
``oracle.chunked``,

    A = strictly_lower(diag(beta) K K^T (.) Gamma),   T = (I + A)^-1,
    R_W = diag(beta gamma) K,  R_U = diag(beta) V,  W = T R_W,  U~ = T R_U,
    U = U~ - W H,   P = (Q K^T (.) Gamma)_{i>=j},
    O = diag(gamma) Q H + P U,   H' = gamma_C H + (diag(dec) K)^T U.

Given dO and dH' (the gradient of the state leaving the chunk), the chain
rule through these definitions, in reverse order, gives

    dU  = P^T dO + diag(dec) K dH'
    dH  = gamma_C dH' + Q^T diag(gamma) dO - W^T dU           (to the previous chunk)
    dP  = (dO U^T)_{i>=j},  dQ = diag(gamma) dO H^T + (dP (.) Gamma) K
    dK~ = U dH'^T,          dW = -dU H^T,   dU~ = dU
    dR_W = T^T dW,  dR_U = T^T dU~,  dV = diag(beta) dR_U
    dT  = dW R_W^T + dU~ R_U^T,  dA = -T^T dT T^T, kept strictly lower
        = -(dR_W W^T + dR_U U~^T), kept strictly lower
    dK  = diag(dec) dK~ + diag(beta gamma) dR_W + (dP (.) Gamma)^T Q
          + diag(beta) D K + D^T diag(beta) K,     D = dA (.) Gamma
    dbeta = rows of dR_U (.) V  +  gamma (.) rows of dR_W (.) K  +  rows of D (.) K K^T
    dG_i  = sum_j E_ij - sum_j E_ji + gamma_i (dgamma_i + beta_i rows(dR_W (.) K)_i)
            - dec_i rows(dK~ (.) K)_i,   plus, for the last token,
            gamma_C <dH', H> + sum_j dec_j rows(dK~ (.) K)_j,
    with E = dP (.) Q K^T (.) Gamma + beta_i D (.) K K^T and dgamma_i = rows(dO H^T (.) Q)_i,
    dg_t = sum_{i >= t} dG_i   (G is a prefix sum of g).

The states H entering each chunk come from the forward recurrence of
``oracle.chunked``; the gradients dH' run backwards over the chunks.

Parity status: pinned (tests/test_oracle_grad_pins.py, chunked-vs-autograd).
"""
from __future__ import annotations

import numpy as np

C = 64


def _one(q, k, v, g, beta, h0, d_o, dhN):
    """One (sequence, head): q, k [L, dk], v, d_o [L, dv], g, beta [L], h0 and
    dhN [dk, dv].  Returns dq, dk, dv, dg, dbeta (per token) and dh0."""
    L, dk = q.shape
    dv = v.shape[1]
    nck = (L + C - 1) // C
    pad = nck * C - L

    def padded(x):
        return np.concatenate([x, np.zeros((pad,) + x.shape[1:])]) if pad else x

    q, k, v, g, beta, d_o = (padded(x) for x in (q, k, v, g, beta, d_o))
    low = np.tril(np.ones((C, C)), -1)
    inc = np.tril(np.ones((C, C)))

    chunks, H = [], h0.copy()
    for c in range(nck):
        s = slice(c * C, (c + 1) * C)
        G = np.cumsum(g[s])
        gam, gC = np.exp(G), np.exp(G[-1])
        Gam = np.exp(G[:, None] - G[None, :]) * inc
        dec = np.exp(G[-1] - G)
        KK, QK = k[s] @ k[s].T, q[s] @ k[s].T
        A = beta[s][:, None] * KK * Gam * low
        T = np.linalg.inv(np.eye(C) + A)
        RW, RU = (beta[s] * gam)[:, None] * k[s], beta[s][:, None] * v[s]
        W, Ut = T @ RW, T @ RU
        P = QK * Gam
        chunks.append(dict(s=s, G=G, gam=gam, gC=gC, Gam=Gam, dec=dec, KK=KK, QK=QK, T=T,
                           RW=RW, RU=RU, W=W, Ut=Ut, P=P, H=H.copy()))
        H = gC * H + (dec[:, None] * k[s]).T @ (Ut - W @ H)

    out = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v))}
    out["dg"], out["dbeta"] = np.zeros(len(g)), np.zeros(len(g))
    dH = dhN.copy()
    for ch in reversed(chunks):
        s, H, T, W, Ut, P, Gam = ch["s"], ch["H"], ch["T"], ch["W"], ch["Ut"], ch["P"], ch["Gam"]
        gam, dec, gC = ch["gam"], ch["dec"], ch["gC"]
        qc, kc, vc, bc, dO = q[s], k[s], v[s], beta[s], d_o[s]
        dHp = dH                                        # gradient of the state leaving
        U = Ut - W @ H
        dU = P.T @ dO + (dec[:, None] * kc) @ dHp
        dH = gC * dHp + (gam[:, None] * qc).T @ dO - W.T @ dU
        dP = (dO @ U.T) * inc
        dOHt = dO @ H.T
        dQ = gam[:, None] * dOHt + (dP * Gam) @ kc
        dKt = U @ dHp.T
        dW = -dU @ H.T
        dRW, dRU = T.T @ dW, T.T @ dU
        dA = -(dRW @ W.T + dRU @ Ut.T) * low
        D = dA * Gam
        dK = (dec[:, None] * dKt + (bc * gam)[:, None] * dRW + (dP * Gam).T @ qc
              + bc[:, None] * (D @ kc) + D.T @ (bc[:, None] * kc))
        dV = bc[:, None] * dRU
        dbg = np.sum(dRW * kc, axis=1)                  # gradient of beta_i gamma_i
        ddec = np.sum(dKt * kc, axis=1)
        dgam = np.sum(dOHt * qc, axis=1) + bc * dbg
        dB = np.sum(dRU * vc, axis=1) + gam * dbg + np.sum(D * ch["KK"], axis=1)
        E = dP * ch["QK"] * Gam + bc[:, None] * D * ch["KK"]
        dG = E.sum(axis=1) - E.sum(axis=0) + gam * dgam - dec * ddec
        dG[-1] += gC * np.sum(dHp * H) + np.sum(dec * ddec)
        out["dq"][s], out["dk"][s], out["dv"][s] = dQ, dK, dV
        out["dbeta"][s] = dB
        out["dg"][s] = np.cumsum(dG[::-1])[::-1]
    res = {n: x[:L] for n, x in out.items()}
    res["dh0"] = dH
    return res


def backward(q, k, v, g, beta, initial_state, d_o, d_final_state=None, cu_seqlens=None):
    """Same interface and result keys (dq, dk, dv, dg, dbeta, dh0) as
    ``oracle.grad.backward``; every array fp64 numpy."""
    def f64(x):
        if x is None:
            return None
        if hasattr(x, "detach"):
            x = x.detach().to("cpu").double().numpy()
        return np.asarray(x, dtype=np.float64)

    q, k, v, g, beta, d_o = (f64(x) for x in (q, k, v, g, beta, d_o))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        bounds = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in (f64(cu_seqlens).astype(np.int64))]
        bounds = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    N = len(bounds)
    h0 = f64(initial_state)
    h0 = np.zeros((N, H, dk, dv)) if h0 is None else h0
    dhN = f64(d_final_state)
    dhN = np.zeros((N, H, dk, dv)) if dhN is None else dhN
    res = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
           "dg": np.zeros_like(g), "dbeta": np.zeros_like(beta), "dh0": np.zeros((N, H, dk, dv))}
    for n, (b, a, e) in enumerate(bounds):
        for h in range(H):
            if e == a:
                res["dh0"][n, h] = dhN[n, h]
                continue
            r = _one(q[b, a:e, h], k[b, a:e, h], v[b, a:e, h], g[b, a:e, h], beta[b, a:e, h],
                     h0[n, h], d_o[b, a:e, h], dhN[n, h])
            for name in ("dq", "dk", "dv", "dg", "dbeta"):
                res[name][b, a:e, h] = r[name]
            res["dh0"][n, h] = r["dh0"]
    return res
