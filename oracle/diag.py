"""Oracle for the HyMo pages' own GDN recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU-baseline leg of ``bench.py`` may use this module;
the product path never imports it, and it imports nothing from the product.

The recurrence, per (batch row, head), token by token in fp64:

    h_t = exp(g_t * A) (.) h_{t-1} + b_t (x) v_t        h_t in R^{S x D}
    o_t = c_t^T h_t                                      o_t in R^D

with A = -exp(A_log[h]) in R^S, one decay rate per state row, and g_t a
positive per-head scalar gate ("Model Architecture Walkthrough", section
5.2.1, the recurrence and its symbol list; "Optimization Quartet", Triton GDN
kernel section 3.2, the shapes v, b, c, g, A_log).  ``exp(g_t * A) (.)``
scales row s of the state by exp(g_t A_s); ``b_t (x) v_t`` is the outer
product.  The read follows the write, as the two lines are written.  There is
no beta and no erase term: this is the pages' form, not the gated delta rule
of the main path.

Parity status: pinned by ``tests/test_oracle_diag_pins.py`` against the
unrolled form of the pages ("Model Architecture Walkthrough", section 5.3.1),
the no-decay limit (linear attention with separate read and write keys, same
page, section 5.2.3) and the scalar-decay mode of the C oracle.

``forward_delta`` is the same per-row decay combined with the delta rule's
erase (the gated delta rule of the main path with its scalar gate replaced by
the pages' diagonal one), token by token in fp64:

    hbar_t = exp(g_t * A) (.) h_{t-1}
    h_t    = hbar_t + beta_t b_t (v_t - hbar_t^T b_t)^T
    o_t    = c_t^T h_t

The decay acts first and the erase reads the decayed state, so that with
beta_t = 1 and a unit b_t the state returns v_t for the key b_t right after
the write (the delta rule's overwrite).  Parity status: pinned by the same
test file against the C oracle's gated delta rule (all rates of a head
equal), pure decay (beta = 0), the overwrite property, decoupled scalar
recursions for basis-vector keys, and chaining.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def forward(v, b, c, g, A_log, initial_state=None):
    """v ``[B, T, H, D]``; b, c ``[B, T, H, S]``; g ``[B, T, H]``; A_log ``[H, S]``;
    initial_state ``[B, H, S, D]`` or None (zeros).  Returns ``(o, final_state)``
    as fp64 arrays: o ``[B, T, H, D]``, final_state ``[B, H, S, D]``."""
    v = _f64(v); b = _f64(b); c = _f64(c); g = _f64(g); A_log = _f64(A_log)
    B, T, H, D = v.shape
    S = b.shape[-1]
    if b.shape != (B, T, H, S) or c.shape != (B, T, H, S) or g.shape != (B, T, H) or \
            A_log.shape != (H, S):
        raise ValueError("diag oracle: shape mismatch")
    A = -np.exp(A_log)                                   # [H, S], negative
    h = np.zeros((B, H, S, D)) if initial_state is None else _f64(initial_state).copy()
    if h.shape != (B, H, S, D):
        raise ValueError("diag oracle: initial_state must be [B, H, S, D]")
    o = np.zeros((B, T, H, D))
    for t in range(T):
        decay = np.exp(g[:, t, :, None] * A[None, :, :])   # [B, H, S]
        h = decay[..., None] * h + b[:, t, :, :, None] * v[:, t, :, None, :]
        o[:, t] = np.einsum("bhs,bhsd->bhd", c[:, t], h)
    return o, h


def forward_delta(v, b, c, g, A_log, beta, initial_state=None):
    """The per-row decay with the delta rule's erase and write strength beta.

    v ``[B, T, H, D]``; b, c ``[B, T, H, S]``; g, beta ``[B, T, H]``; A_log
    ``[H, S]``; initial_state ``[B, H, S, D]`` or None (zeros).  Returns
    ``(o, final_state)`` as fp64 arrays shaped like ``forward``'s."""
    v = _f64(v); b = _f64(b); c = _f64(c); g = _f64(g); A_log = _f64(A_log)
    beta = _f64(beta)
    B, T, H, D = v.shape
    S = b.shape[-1]
    if b.shape != (B, T, H, S) or c.shape != (B, T, H, S) or g.shape != (B, T, H) or \
            beta.shape != (B, T, H) or A_log.shape != (H, S):
        raise ValueError("diag delta oracle: shape mismatch")
    A = -np.exp(A_log)                                   # [H, S], negative
    h = np.zeros((B, H, S, D)) if initial_state is None else _f64(initial_state).copy()
    if h.shape != (B, H, S, D):
        raise ValueError("diag delta oracle: initial_state must be [B, H, S, D]")
    o = np.zeros((B, T, H, D))
    for t in range(T):
        decay = np.exp(g[:, t, :, None] * A[None, :, :])             # [B, H, S]
        hbar = decay[..., None] * h                                   # rows scaled
        bt = b[:, t]                                                  # [B, H, S]
        pred = np.einsum("bhs,bhsd->bhd", bt, hbar)                   # hbar^T b
        err = beta[:, t, :, None] * (v[:, t] - pred)                  # [B, H, D]
        h = hbar + bt[..., None] * err[:, :, None, :]
        o[:, t] = np.einsum("bhs,bhsd->bhd", c[:, t], h)
    return o, h
