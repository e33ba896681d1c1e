"""Oracle for the GDN block's prologue and epilogue -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU-baseline leg of ``bench.py`` may use this module;
the product path never imports it, and it imports nothing from the product.
Everything is fp64 numpy, written from the definitions:

``conv_silu``   causal depthwise conv1d then SiLU ("Model Architecture
                Walkthrough", section 5.4.1: depthwise Conv1d with d_conv taps
                and padding d_conv - 1, tail trimmed; section 5.5, step 2).
``epilogue``    skip and output gate of the block: (o + D v) * g_gate
                (same page, section 5.5, step 6).
``sigmoid``     the gate nonlinearity g = sigmoid(dt) (section 5.2.1).

Parity status: pinned by ``tests/test_oracle_block_pins.py`` (PyTorch's own
conv1d and SiLU on the CPU, impulse responses, chaining, closed forms and
planted mistakes).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def sigmoid(z):
    z = _f64(z)
    return 1.0 / (1.0 + np.exp(-z))


def conv_silu(x, w, x_prev=None):
    """x ``[B, T, C]``; w ``[C, K]`` (tap k multiplies x[t - (K - 1) + k]);
    x_prev ``[B, K-1, C]`` or None (zeros before token 0).  Returns
    ``(y, x_tail)``: y ``[B, T, C]`` = silu(conv), x_tail ``[B, K-1, C]`` the
    last K-1 inputs of x_prev followed by x."""
    x = _f64(x); w = _f64(w)
    B, T, C = x.shape
    K = w.shape[1]
    prev = np.zeros((B, K - 1, C)) if x_prev is None else _f64(x_prev)
    xs = np.concatenate([prev, x], axis=1)            # token t of x is row t + K - 1
    z = np.zeros((B, T, C))
    for k in range(K):
        z += w[None, None, :, k] * xs[:, k:k + T, :]
    y = z * sigmoid(z)
    return y, xs[:, xs.shape[1] - (K - 1):, :]


def epilogue(o, v, D, g_gate):
    """o, v ``[B, T, H, Dh]``; D ``[H]``; g_gate ``[B, T, H]``: (o + D v) * g_gate."""
    o = _f64(o); v = _f64(v); D = _f64(D); g_gate = _f64(g_gate)
    return (o + D[None, None, :, None] * v) * g_gate[..., None]
