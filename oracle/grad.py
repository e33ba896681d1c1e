"""Oracle for the backward pass of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU-baseline leg of ``bench.py`` may use this module;
the product path never imports it, and it imports nothing from the product.

``backward`` writes the forward recurrence token by token in fp64 PyTorch on
the CPU, in the transposed-state form the library uses (H = S^T, dk x dv):

    H_t = alpha_t H_{t-1} (I - beta_t k_t k_t^T)^T ... written out as
    H_t = alpha_t (H_{t-1} - beta_t k_t (k_t^T H_{t-1})) + beta_t k_t v_t^T,
    o_t = H_t^T q_t,   alpha_t = exp(g_t)

(the gated delta rule of Yang et al., arXiv 2412.06464, named by "v1.0
Architecture & Design Spec", section 2.3; the pages' own kernel ships a
backward: "Optimization Quartet", Triton GDN kernel section 3.4, and "Model
Architecture Walkthrough", section 6.5 -- backpropagation through time).  It
then lets torch.autograd differentiate the scalar
sum(o * d_o) + sum(H_N * d_final_state), which gives the vector-Jacobian
products dq, dk, dv, dg, dbeta and d_initial_state.

Parity status: pinned by ``tests/test_oracle_grad_pins.py`` -- central finite
differences of the independent C oracle's forward, the beta = 0 closed form,
and planted mistakes.
"""
from __future__ import annotations

import numpy as np
import torch


def _t(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        return x.detach().to("cpu").double().clone()
    return torch.from_numpy(np.asarray(x, dtype=np.float64).copy())


def backward(q, k, v, g, beta, initial_state, d_o, d_final_state=None, cu_seqlens=None):
    """Shapes as the library: q, k ``[B, T, H, dk]``, v ``[B, T, H, dv]``, g, beta
    ``[B, T, H]``, initial_state ``[N, H, dk, dv]`` or None, d_o like v,
    d_final_state ``[N, H, dk, dv]`` or None; cu_seqlens (B = 1) or None.
    Returns a dict of fp64 numpy arrays dq, dk, dv, dg, dbeta, dh0 (dh0 is
    zeros when there is no initial state) and the forward o, final_state."""
    q, k, v, g, beta = _t(q), _t(k), _t(v), _t(g), _t(beta)
    d_o = _t(d_o)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        bounds = [(n, 0, T) for n in range(B)]
    else:
        cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        bounds = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    N = len(bounds)
    h0 = _t(initial_state) if initial_state is not None else torch.zeros(N, H, dk, dv,
                                                                          dtype=torch.float64)
    dhN = _t(d_final_state)
    leaves = [q, k, v, g, beta, h0]
    for x in leaves:
        x.requires_grad_(True)
    zero = torch.zeros(H, dv, dtype=torch.float64)
    o_rows = [[zero] * T for _ in range(B)]
    finals = []
    for n, (row, s, e) in enumerate(bounds):
        Hs = h0[n]                                                  # [H, dk, dv]
        for t in range(s, e):
            kt, vt, qt = k[row, t], v[row, t], q[row, t]            # [H, dk], [H, dv], [H, dk]
            a = torch.exp(g[row, t])[:, None, None]
            bt = beta[row, t][:, None, None]
            kH = torch.einsum("hk,hkv->hv", kt, Hs)                 # k^T H_{t-1}
            Hs = a * (Hs - bt * kt[:, :, None] * kH[:, None, :]) + bt * kt[:, :, None] * vt[:, None, :]
            o_rows[row][t] = torch.einsum("hkv,hk->hv", Hs, qt)
        finals.append(Hs)
    o = torch.stack([torch.stack(r) for r in o_rows])
    hN = torch.stack(finals)
    loss = (o * d_o).sum()
    if dhN is not None:
        loss = loss + (hN * dhN).sum()
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    names = ["dq", "dk", "dv", "dg", "dbeta", "dh0"]
    res = {}
    for name, gr, leaf in zip(names, grads, leaves):
        res[name] = (torch.zeros_like(leaf) if gr is None else gr).detach().numpy()
    res["o"] = o.detach().numpy()
    res["final_state"] = hN.detach().numpy()
    return res
