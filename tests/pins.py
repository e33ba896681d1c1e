"""Pins for the oracle: checks against facts that the mathematics of the gated
delta rule fixes, independent of any implementation of it.

Each ``pin_*`` function takes a ``forward`` callable with the signature of
``oracle.forward`` and returns a list of ``(label, error, bound)``; a pin holds
when every error is within its bound.  ``tests/test_oracle_pins.py`` runs them
on the oracle; ``tests/test_oracle_mutants.py`` plants plausible mistakes in a
copy of the oracle's C source and checks that some pin catches each one.

Recurrence (transposed-state form used by the library, H = S^T):
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t
(gated delta rule, Yang et al. arXiv 2412.06464, named in "v1.0 Architecture &
Design Spec" section 2.3).
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel(a, b) -> float:
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def _rand_unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _inputs(rng, B, T, H, dk, dv, gate_scale=0.5):
    q = _rand_unit_rows(rng, (B, T, H, dk))
    k = _rand_unit_rows(rng, (B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H)))) * gate_scale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    return q, k, v, g, beta


# --------------------------------------------------------------------------
# Hand-derived two-token example (tests/golden/two_token_hand.json)
# --------------------------------------------------------------------------
def pin_golden_two_token(forward):
    with open(os.path.join(GOLDEN, "two_token_hand.json")) as f:
        gold = json.load(f)
    q = np.array(gold["q"])[None, :, None, :]
    k = np.array(gold["k"])[None, :, None, :]
    v = np.array(gold["v"])[None, :, None, :]
    g = np.log(np.array(gold["alpha"]))[None, :, None]
    beta = np.array(gold["beta"])[None, :, None]
    o, sN = forward(q, k, v, g, beta)
    return [("golden o", rel(o[0, :, 0], gold["o"]), 1e-13),
            ("golden final_state", rel(sN[0, 0], gold["final_state_dk_by_dv"]), 1e-13)]


# --------------------------------------------------------------------------
# P1: beta = 0 leaves only the decay -- closed-form cumulative decay
# ("Model Architecture Walkthrough" section 5.3.1: weight = exp(sum of gates))
# --------------------------------------------------------------------------
def pin_beta_zero_closed_form(forward, seed=1):
    rng = np.random.default_rng(seed)
    B, T, H, dk, dv = 2, 45, 3, 5, 3
    q, k, v, g, _ = _inputs(rng, B, T, H, dk, dv)
    beta = np.zeros((B, T, H))
    H0 = rng.standard_normal((B, H, dk, dv))
    o, sN = forward(q, k, v, g, beta, H0)
    G = np.cumsum(g, axis=1)                                   # [B,T,H]
    o_ref = np.exp(G)[..., None] * np.einsum("bhkd,bthk->bthd", H0, q)
    s_ref = np.exp(G[:, -1])[..., None, None] * H0
    return [("beta=0 o", rel(o, o_ref), 1e-12),
            ("beta=0 final_state", rel(sN, s_ref), 1e-12)]


# --------------------------------------------------------------------------
# P2: erase-off, beta-free recurrence (the pages' printed GDN form with b=k,
# c=q and a scalar decay) against its unrolled closed form; g = 0 gives plain
# linear attention ("Model Architecture Walkthrough" sections 5.1.2, 5.2.3, 5.3.1)
# --------------------------------------------------------------------------
def pin_gla_closed_form(forward_gla, seed=2):
    rng = np.random.default_rng(seed)
    B, T, H, dk, dv = 1, 30, 2, 4, 6
    q, k, v, g, _ = _inputs(rng, B, T, H, dk, dv)
    H0 = rng.standard_normal((B, H, dk, dv))
    out = []
    for label, gg in (("gla", g), ("linear attention (g=0)", np.zeros_like(g))):
        o, sN = forward_gla(q, k, v, gg, None, H0)
        G = np.cumsum(gg, axis=1)
        o_ref = np.zeros_like(o)
        for h in range(H):
            for t in range(T):
                acc = np.exp(G[0, t, h]) * (H0[0, h].T @ q[0, t, h])
                for s in range(t + 1):
                    acc = acc + np.exp(G[0, t, h] - G[0, s, h]) * \
                        (k[0, s, h] @ q[0, t, h]) * v[0, s, h]
                o_ref[0, t, h] = acc
        out.append((label + " o", rel(o, o_ref), 1e-12))
    return out


# --------------------------------------------------------------------------
# P3: alpha = 1, beta = 1, orthonormal keys -> exact overwrite (delta rule)
# --------------------------------------------------------------------------
def pin_exact_overwrite(forward, seed=3):
    rng = np.random.default_rng(seed)
    dk, dv = 6, 4
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm.T                                   # rows orthonormal
    vals = rng.standard_normal((dk, dv))
    vnew = rng.standard_normal(dv)
    a = 2
    # tokens: write all dk keys, then rewrite key a, then read every key back
    ks = np.concatenate([keys, keys[a:a + 1], np.zeros((dk, dk))])
    vs = np.concatenate([vals, vnew[None], np.zeros((dk, dv))])
    qs = np.concatenate([keys, keys[a:a + 1], keys])
    betas = np.concatenate([np.ones(dk + 1), np.zeros(dk)])
    T = len(ks)
    H0 = rng.standard_normal((1, 1, dk, dv))
    o, sN = forward(qs[None, :, None], ks[None, :, None], vs[None, :, None],
                    np.zeros((1, T, 1)), betas[None, :, None], H0)
    o = o[0, :, 0]
    expect_written = vals.copy()
    expect_written[a] = vnew
    out = [
        # after writing key s, reading key s returns v_s exactly
        ("overwrite read-after-write", rel(o[:dk], vals), 1e-12),
        ("overwrite rewrite", rel(o[dk], vnew), 1e-12),
        # final read-back: every key returns its latest value
        ("overwrite read-back", rel(o[dk + 1:], expect_written), 1e-12),
        # the initial state is fully erased: H = sum_s k_s v_s^T
        ("overwrite final_state", rel(sN[0, 0], keys.T @ expect_written), 1e-12),
    ]
    return out


# --------------------------------------------------------------------------
# P4: chunked WY/UT form == sequential form, for several chunk sizes
# --------------------------------------------------------------------------
def pin_chunked_equals_sequential(forward, chunked_forward, seed=4):
    rng = np.random.default_rng(seed)
    out = []
    B, T, H, dk, dv = 1, 200, 2, 16, 24
    q, k, v, g, beta = _inputs(rng, B, T, H, dk, dv, gate_scale=1.0)
    H0 = 0.1 * rng.standard_normal((B, H, dk, dv))
    o_s, s_s = forward(q, k, v, g, beta, H0)
    for C in (1, 2, 16, 37, 64):
        o_c, s_c = chunked_forward(q, k, v, g, beta, H0, chunk_size=C)
        out.append((f"chunked C={C} o", rel(o_c, o_s), 1e-12))
        out.append((f"chunked C={C} final_state", rel(s_c, s_s), 1e-12))
    # packed sequences, chunking restarting at each sequence start
    cu = np.array([0, 5, 70, 71, 200])
    H0v = 0.1 * rng.standard_normal((4, H, dk, dv))
    o_s, s_s = forward(q, k, v, g, beta, H0v, cu)
    o_c, s_c = chunked_forward(q, k, v, g, beta, H0v, cu, chunk_size=64)
    out.append(("chunked varlen o", rel(o_c, o_s), 1e-12))
    out.append(("chunked varlen final_state", rel(s_c, s_s), 1e-12))
    return out


# --------------------------------------------------------------------------
# P5: running [0, T1) then [T1, T) with final -> initial equals one run
# --------------------------------------------------------------------------
def pin_state_chaining(forward, seed=5):
    rng = np.random.default_rng(seed)
    B, T, H, dk, dv = 2, 90, 2, 8, 5
    q, k, v, g, beta = _inputs(rng, B, T, H, dk, dv)
    H0 = rng.standard_normal((B, H, dk, dv))
    o, s = forward(q, k, v, g, beta, H0)
    T1 = 37
    o1, s1 = forward(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], H0)
    o2, s2 = forward(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], s1)
    return [("chaining o", rel(np.concatenate([o1, o2], axis=1), o), 1e-14),
            ("chaining final_state", rel(s2, s), 1e-14)]


# --------------------------------------------------------------------------
# P6: exact rational brute force of the unrolled product on tiny inputs
#   S_t = S_0 prod_{r<=t} M_r + sum_{s<=t} beta_s v_s k_s^T prod_{s<r<=t} M_r,
#   M_r = alpha_r (I - beta_r k_r k_r^T)   (products in increasing time order)
# --------------------------------------------------------------------------
def _fmat(rows, cols, val=Fraction(0)):
    return [[val for _ in range(cols)] for _ in range(rows)]


def _fmul(A, B):
    return [[sum((A[i][p] * B[p][j] for p in range(len(B))), Fraction(0))
             for j in range(len(B[0]))] for i in range(len(A))]


def _fadd(A, B):
    return [[A[i][j] + B[i][j] for j in range(len(A[0]))] for i in range(len(A))]


def _fscale(c, A):
    return [[c * x for x in row] for row in A]


def brute_force_exact(alpha, beta, q, k, v, S0):
    """Unrolled-product evaluation in exact rationals; returns (o[t][j], S_T)."""
    T = len(alpha)
    dk = len(k[0]); dv = len(v[0])
    eye = [[Fraction(int(i == j)) for j in range(dk)] for i in range(dk)]
    M = []
    for t in range(T):
        kk = [[k[t][i] * k[t][j] for j in range(dk)] for i in range(dk)]
        M.append(_fscale(alpha[t], _fadd(eye, _fscale(-beta[t], kk))))
    outs = []
    S_t = None
    for t in range(T):
        def prod(lo, hi):  # M_lo M_{lo+1} ... M_hi (identity if empty)
            P = eye
            for r in range(lo, hi + 1):
                P = _fmul(P, M[r])
            return P
        S_t = _fmul(S0, prod(0, t))
        for s in range(t + 1):
            vk = [[beta[s] * v[s][i] * k[s][j] for j in range(dk)] for i in range(dv)]
            S_t = _fadd(S_t, _fmul(vk, prod(s + 1, t)))
        outs.append([sum((S_t[i][j] * q[t][j] for j in range(dk)), Fraction(0))
                     for i in range(dv)])
    return outs, S_t


def pin_brute_force(forward, seed=6):
    rng = np.random.default_rng(seed)
    out = []
    for (T, dk, dv) in ((1, 2, 2), (4, 2, 3), (6, 3, 2), (5, 3, 3)):
        dy = lambda shape: rng.integers(-8, 9, shape) / 8       # dyadic rationals
        q, k, v = dy((T, dk)), dy((T, dk)), dy((T, dv))
        S0 = dy((dv, dk))
        alpha = [Fraction(int(a), 16) for a in rng.integers(1, 17, T)]
        beta = [Fraction(int(b), 8) for b in rng.integers(0, 9, T)]
        fq = [[Fraction(x) for x in row] for row in q]
        fk = [[Fraction(x) for x in row] for row in k]
        fv = [[Fraction(x) for x in row] for row in v]
        fS0 = [[Fraction(x) for x in row] for row in S0]
        o_ex, S_ex = brute_force_exact(alpha, beta, fq, fk, fv, fS0)
        o, sN = forward(q[None, :, None], k[None, :, None], v[None, :, None],
                        np.log(np.array([float(a) for a in alpha]))[None, :, None],
                        np.array([float(b) for b in beta])[None, :, None],
                        S0.T[None, None])
        o_ex = np.array([[float(x) for x in row] for row in o_ex])
        S_ex = np.array([[float(x) for x in row] for row in S_ex])
        out.append((f"brute T={T} dk={dk} dv={dv} o", rel(o[0, :, 0], o_ex), 1e-13))
        out.append((f"brute T={T} dk={dk} dv={dv} final_state",
                    rel(sN[0, 0], S_ex.T), 1e-13))
    return out


# --------------------------------------------------------------------------
# P7: invariants -- non-expansive carry (alpha = 1, |k| = 1, beta in (0,1]):
# I - beta k k^T has eigenvalues {1, 1 - beta}, so ||S_t|| <= ||S_{t-1}|| + beta ||v_t||;
# and packed sequences equal separate runs, bit for bit.
# --------------------------------------------------------------------------
def pin_nonexpansive(forward, seed=7):
    rng = np.random.default_rng(seed)
    dk, dv, T = 6, 4, 40
    q, k, v, _, beta = _inputs(rng, 1, T, 1, dk, dv)
    S = rng.standard_normal((1, 1, dk, dv))
    worst = 0.0
    for t in range(T):
        sl = slice(t, t + 1)
        _, S_new = forward(q[:, sl], k[:, sl], v[:, sl], np.zeros((1, 1, 1)),
                           beta[:, sl], S)
        lhs = np.linalg.norm(S_new[0, 0], 2)
        rhs = np.linalg.norm(S[0, 0], 2) + beta[0, t, 0] * np.linalg.norm(v[0, t, 0])
        worst = max(worst, (lhs - rhs) / rhs)
        S = S_new
    return [("non-expansive carry (excess)", max(worst, 0.0), 1e-12)]


def pin_varlen_bitwise(forward, seed=8):
    rng = np.random.default_rng(seed)
    lens = [3, 64, 65, 1, 130]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1]); H, dk, dv = 2, 8, 12
    q, k, v, g, beta = _inputs(rng, 1, T, H, dk, dv)
    H0 = rng.standard_normal((len(lens), H, dk, dv))
    o, s = forward(q, k, v, g, beta, H0, cu)
    worst = 0.0
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        o1, s1 = forward(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], H0[n:n + 1])
        worst = max(worst, float(np.max(np.abs(o1 - o[:, a:b]))),
                    float(np.max(np.abs(s1 - s[n:n + 1]))))
    return [("varlen == separate runs (max abs diff)", worst, 0.0)]


def run(pins):
    """Flatten pin results; return the failing entries."""
    return [(lab, err, bound) for lab, err, bound in pins if not err <= bound]
