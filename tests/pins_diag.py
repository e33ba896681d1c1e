"""Pins for the diagonal-decay oracle (``oracle.diag``): facts the pages and
the mathematics fix for the HyMo recurrence

    h_t = exp(g_t A) (.) h_{t-1} + b_t (x) v_t,   o_t = c_t^T h_t,   A = -exp(A_log)

("Model Architecture Walkthrough", section 5.2.1).  Each ``pin_*`` takes a
``forward`` with the signature of ``oracle.diag.forward`` and returns a list of
``(label, error, bound)``; ``pins.run`` lists the violated ones.
"""
from __future__ import annotations

import json
import os

import numpy as np

from pins import GOLDEN, rel


def inputs(rng, B, T, H, S, D, A_log_const=False):
    """Gates in (0, 1) (a sigmoid, as the pages' g is), keys and values N(0, 1)."""
    v = rng.standard_normal((B, T, H, D))
    b = rng.standard_normal((B, T, H, S))
    c = rng.standard_normal((B, T, H, S))
    g = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    if A_log_const:
        A_log = np.repeat(rng.uniform(-2.0, 1.0, (H, 1)), S, axis=1)
    else:
        A_log = rng.uniform(-2.0, 1.0, (H, S))
    return v, b, c, g, A_log


# --------------------------------------------------------------------------
# Golden: the per-step decay factors the pages print (section 5.3.2)
# --------------------------------------------------------------------------
def pin_golden_page_decay(forward):
    with open(os.path.join(GOLDEN, "diag_decay_pages.json")) as f:
        gold = json.load(f)
    out = []
    for case in gold["cases"]:
        # S = D = 1, b = c = v = 1, g = 1 twice: o_1 = 1, o_2 = decay + 1
        one = np.ones((1, 2, 1, 1))
        g = np.full((1, 2, 1), case["g"])
        o, _ = forward(one, one, one, g, np.array([[case["A_log"]]]))
        decay = o[0, 1, 0, 0] - o[0, 0, 0, 0]
        out.append((f"page decay A_log={case['A_log']:.3f}",
                    abs(decay - case["decay"]) / case["tolerance"], 1.0))
    return out


# --------------------------------------------------------------------------
# Unrolled closed form (section 5.3.1): the contribution of token k to h_t is
# weighted by exp(A * sum_{j=k+1..t} g_j); h_0 by exp(A * sum_{j<=t} g_j).
# --------------------------------------------------------------------------
def unrolled(v, b, c, g, A_log, h0):
    B, T, H, D = v.shape
    S = b.shape[-1]
    A = -np.exp(A_log)
    o = np.zeros((B, T, H, D))
    for bb in range(B):
        for hh in range(H):
            for t in range(T):
                h = np.exp(A[hh] * g[bb, :t + 1, hh].sum())[:, None] * h0[bb, hh]
                for k in range(t + 1):
                    w = np.exp(A[hh] * g[bb, k + 1:t + 1, hh].sum())      # [S]
                    h = h + w[:, None] * np.outer(b[bb, k, hh], v[bb, k, hh])
                o[bb, t, hh] = c[bb, t, hh] @ h
    # final state: the same sums at t = T - 1
    hN = np.zeros((B, H, S, D))
    for bb in range(B):
        for hh in range(H):
            h = np.exp(A[hh] * g[bb, :, hh].sum())[:, None] * h0[bb, hh]
            for k in range(T):
                w = np.exp(A[hh] * g[bb, k + 1:, hh].sum())
                h = h + w[:, None] * np.outer(b[bb, k, hh], v[bb, k, hh])
            hN[bb, hh] = h
    return o, hN


def pin_unrolled(forward, seed=11):
    rng = np.random.default_rng(seed)
    out = []
    for (B, T, H, S, D) in ((2, 23, 2, 3, 3), (1, 17, 3, 4, 5)):
        v, b, c, g, A_log = inputs(rng, B, T, H, S, D)
        h0 = rng.standard_normal((B, H, S, D))
        o, hN = forward(v, b, c, g, A_log, h0)
        o_ref, h_ref = unrolled(v, b, c, g, A_log, h0)
        out += [(f"unrolled o S={S} D={D}", rel(o, o_ref), 1e-12),
                (f"unrolled final S={S} D={D}", rel(hN, h_ref), 1e-12)]
    return out


# --------------------------------------------------------------------------
# No decay, b = c = k: plain linear attention, o_t = sum_{j<=t} (k_t . k_j) v_j
# (section 5.2.3: linear attention is the special case b = c = k, no gating)
# --------------------------------------------------------------------------
def pin_linear_attention(forward, seed=12):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 2, 19, 2, 4, 3
    v, k, _, g, _ = inputs(rng, B, T, H, S, D)
    A_log = np.full((H, S), -1000.0)     # A = -exp(-1000) = -0.0: factor exactly 1
    o, hN = forward(v, k, k, g, A_log)
    o_ref = np.zeros_like(v)
    for t in range(T):
        w = np.einsum("bhs,bjhs->bjh", k[:, t], k[:, :t + 1])           # [B, t+1, H]
        o_ref[:, t] = np.einsum("bjh,bjhd->bhd", w, v[:, :t + 1])
    h_ref = np.einsum("bjhs,bjhd->bhsd", k, v)
    return [("linear attention o", rel(o, o_ref), 1e-12),
            ("linear attention final", rel(hN, h_ref), 1e-12)]


# --------------------------------------------------------------------------
# A_log constant over the state rows: a scalar decay exp(g_t A) per head, i.e.
# the erase-free scalar-gate recurrence of the sequential C oracle with
# q = c, k = b and natural-log gate g_t * A.
# --------------------------------------------------------------------------
def pin_scalar_decay(forward, forward_gla, seed=13):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 2, 21, 3, 5, 4
    v, b, c, g, A_log = inputs(rng, B, T, H, S, D, A_log_const=True)
    h0 = rng.standard_normal((B, H, S, D))
    o, hN = forward(v, b, c, g, A_log, h0)
    A = -np.exp(A_log[:, 0])                                             # [H]
    o2, h2 = forward_gla(c, b, v, g * A[None, None, :], None, h0)
    return [("scalar decay o", rel(o, o2), 1e-12), ("scalar decay final", rel(hN, h2), 1e-12)]


# --------------------------------------------------------------------------
# The rows of the state evolve independently: the output is the sum over s of
# the outputs of the S = 1 problems, one per state row.
# --------------------------------------------------------------------------
def pin_row_independence(forward, seed=14):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 1, 15, 2, 4, 4
    v, b, c, g, A_log = inputs(rng, B, T, H, S, D)
    h0 = rng.standard_normal((B, H, S, D))
    o, hN = forward(v, b, c, g, A_log, h0)
    o_sum = np.zeros_like(o)
    h_rows = np.zeros_like(hN)
    for s in range(S):
        os_, hs = forward(v, b[..., s:s + 1], c[..., s:s + 1], g, A_log[:, s:s + 1],
                          h0[:, :, s:s + 1])
        o_sum += os_
        h_rows[:, :, s] = hs[:, :, 0]
    return [("row sum o", rel(o, o_sum), 1e-12), ("row final", rel(hN, h_rows), 1e-12)]


# --------------------------------------------------------------------------
# Two calls chained through the state equal one call.
# --------------------------------------------------------------------------
def pin_chaining(forward, seed=15):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 2, 26, 2, 3, 5
    v, b, c, g, A_log = inputs(rng, B, T, H, S, D)
    h0 = rng.standard_normal((B, H, S, D))
    o, hN = forward(v, b, c, g, A_log, h0)
    m = 11
    o1, h1 = forward(v[:, :m], b[:, :m], c[:, :m], g[:, :m], A_log, h0)
    o2, h2 = forward(v[:, m:], b[:, m:], c[:, m:], g[:, m:], A_log, h1)
    return [("chained o", rel(np.concatenate([o1, o2], axis=1), o), 1e-13),
            ("chained final", rel(h2, hN), 1e-13)]


# ==========================================================================
# The per-row decay combined with the delta rule (``oracle.diag.forward_delta``):
#   hbar = exp(g_t A) (.) h,  h_t = hbar + beta_t b_t (v_t - hbar^T b_t)^T,  o_t = c_t^T h_t
# ==========================================================================
def delta_inputs(rng, B, T, H, S, D, A_log_const=False):
    """Unit write keys (the delta rule's erase is a projection for beta <= 1
    then), read keys and values N(0, 1), beta in (0, 1), gates in (0, 1)."""
    v, b, c, g, A_log = inputs(rng, B, T, H, S, D, A_log_const)
    b = b / np.linalg.norm(b, axis=-1, keepdims=True)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    return v, b, c, g, A_log, beta


# All rates of a head equal: a scalar decay exp(g_t A) per head, i.e. the
# gated delta rule of the sequential C oracle with q = c, k = b and the
# natural-log gate g_t * A (an independent implementation in C).
def pin_delta_scalar_rates(forward_delta, forward_gdn, seed=21):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 2, 23, 3, 6, 5
    v, b, c, g, A_log, beta = delta_inputs(rng, B, T, H, S, D, A_log_const=True)
    h0 = rng.standard_normal((B, H, S, D))
    o, hN = forward_delta(v, b, c, g, A_log, beta, h0)
    A = -np.exp(A_log[:, 0])                                             # [H]
    o2, h2 = forward_gdn(c, b, v, g * A[None, None, :], beta, h0)
    return [("delta scalar rates o", rel(o, o2), 1e-12),
            ("delta scalar rates final", rel(hN, h2), 1e-12)]


# beta = 0: no erase and no write, only the decay: row s of h_t is
# exp(A_s sum_{j<=t} g_j) times row s of h_0.
def pin_delta_pure_decay(forward_delta, seed=22):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 2, 17, 2, 5, 4
    v, b, c, g, A_log, beta = delta_inputs(rng, B, T, H, S, D)
    h0 = rng.standard_normal((B, H, S, D))
    o, hN = forward_delta(v, b, c, g, A_log, np.zeros_like(beta), h0)
    A = -np.exp(A_log)                                                   # [H, S]
    Gc = np.cumsum(g, axis=1)                                            # [B, T, H]
    scale = np.exp(Gc[..., None] * A[None, None])                        # [B, T, H, S]
    o_ref = np.einsum("bths,bhsd->bthd", c * scale, h0)
    h_ref = scale[:, -1, :, :, None] * h0
    return [("delta pure decay o", rel(o, o_ref), 1e-12),
            ("delta pure decay final", rel(hN, h_ref), 1e-12)]


# The delta rule's overwrite: with beta_t = 1 and a unit key b_t, reading the
# state with c_t = b_t right after the write returns v_t, whatever the state
# held and however its rows decayed.
def pin_delta_overwrite(forward_delta, seed=23):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 2, 19, 2, 6, 4
    v, b, c, g, A_log, beta = delta_inputs(rng, B, T, H, S, D)
    h0 = rng.standard_normal((B, H, S, D))
    o, _ = forward_delta(v, b, b, g, A_log, np.ones_like(beta), h0)
    return [("delta overwrite", rel(o, v), 1e-12)]


# Basis-vector write keys b_t = e_{s_t} decouple the rows: row r decays by
# d_r = exp(g_t A_r) and, when r = s_t, becomes (1 - beta_t) d_r h_r + beta_t v_t.
def pin_delta_basis_keys(forward_delta, seed=24):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 1, 25, 2, 4, 3
    v, _, c, g, A_log, beta = delta_inputs(rng, B, T, H, S, D)
    sel = rng.integers(0, S, size=(B, T, H))
    b = np.zeros((B, T, H, S))
    for bb in range(B):
        for t in range(T):
            for hh in range(H):
                b[bb, t, hh, sel[bb, t, hh]] = 1.0
    h0 = rng.standard_normal((B, H, S, D))
    o, hN = forward_delta(v, b, c, g, A_log, beta, h0)
    A = -np.exp(A_log)
    o_ref = np.zeros_like(o)
    h_ref = np.zeros_like(hN)
    for bb in range(B):
        for hh in range(H):
            rows = [h0[bb, hh, r].copy() for r in range(S)]
            for t in range(T):
                for r in range(S):
                    d = np.exp(g[bb, t, hh] * A[hh, r])
                    if r == sel[bb, t, hh]:
                        rows[r] = (1.0 - beta[bb, t, hh]) * d * rows[r] + beta[bb, t, hh] * v[bb, t, hh]
                    else:
                        rows[r] = d * rows[r]
                o_ref[bb, t, hh] = sum(c[bb, t, hh, r] * rows[r] for r in range(S))
            for r in range(S):
                h_ref[bb, hh, r] = rows[r]
    return [("delta basis keys o", rel(o, o_ref), 1e-12),
            ("delta basis keys final", rel(hN, h_ref), 1e-12)]


def pin_delta_chaining(forward_delta, seed=25):
    rng = np.random.default_rng(seed)
    B, T, H, S, D = 2, 24, 2, 4, 5
    v, b, c, g, A_log, beta = delta_inputs(rng, B, T, H, S, D)
    h0 = rng.standard_normal((B, H, S, D))
    o, hN = forward_delta(v, b, c, g, A_log, beta, h0)
    m = 9
    o1, h1 = forward_delta(v[:, :m], b[:, :m], c[:, :m], g[:, :m], A_log, beta[:, :m], h0)
    o2, h2 = forward_delta(v[:, m:], b[:, m:], c[:, m:], g[:, m:], A_log, beta[:, m:], h1)
    return [("delta chained o", rel(np.concatenate([o1, o2], axis=1), o), 1e-13),
            ("delta chained final", rel(h2, hN), 1e-13)]


def all_delta_pins(forward_delta, forward_gdn):
    res = []
    res += pin_delta_scalar_rates(forward_delta, forward_gdn)
    res += pin_delta_pure_decay(forward_delta)
    res += pin_delta_overwrite(forward_delta)
    res += pin_delta_basis_keys(forward_delta)
    res += pin_delta_chaining(forward_delta)
    return res


def all_pins(forward, forward_gla):
    res = []
    res += pin_golden_page_decay(forward)
    res += pin_unrolled(forward)
    res += pin_linear_attention(forward)
    res += pin_scalar_decay(forward, forward_gla)
    res += pin_row_independence(forward)
    res += pin_chaining(forward)
    return res
