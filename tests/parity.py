"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs, and measure the relative L2 error."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from linear_attention_recurrence_gated_gb300 import gdn as G

# Relative L2 bounds: fp32 storage 1e-4 (o and final state); bf16 storage
# 1e-2 on o and 5e-3 on the final state.
TOL = {torch.float32: (1e-4, 1e-4), torch.bfloat16: (1e-2, 5e-3)}


def rel(a, b) -> float:
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def worst_unit_o(a, b, cu=None) -> float:
    """Largest relative L2 over the (sequence, head) units of an output
    ``[B, T, H, dv]`` (packed sequences: B = 1 and ``cu`` the offsets)."""
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    worst = 0.0
    if cu is None:
        for n in range(a.shape[0]):
            for h in range(a.shape[2]):
                worst = max(worst, rel(a[n, :, h], b[n, :, h]))
    else:
        cu = [int(x) for x in cu]
        for n in range(len(cu) - 1):
            for h in range(a.shape[2]):
                worst = max(worst, rel(a[0, cu[n]:cu[n + 1], h], b[0, cu[n]:cu[n + 1], h]))
    return worst


def worst_unit_state(a, b) -> float:
    """Largest relative L2 over the (sequence, head) units of a state ``[N, H, dk, dv]``."""
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return max(rel(a[n, h], b[n, h]) for n in range(a.shape[0]) for h in range(a.shape[1]))


# Margins of the full-size workloads, printed at the end of the pytest run
# (tests/conftest.py) so that they appear in the tail of its log.
MARGINS = []


def to_dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_forward(inp, **kw):
    d = to_dev(inp)
    o, s = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                     d["cu_seqlens"], check=True, **kw)
    torch.cuda.synchronize()
    return o, s


def oracle_forward(inp, **kw):
    return oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                          inp["initial_state"], inp["cu_seqlens"], **kw)


def compare(inp, gpu_kw=None, oracle_kw=None, units=False):
    """Return (rel_o, rel_state, o_gpu, s_gpu) for one input set; with
    ``units`` also the worst (sequence, head) unit of each:
    (rel_o, rel_state, o_gpu, s_gpu, worst_o, worst_state)."""
    o, s = gpu_forward(inp, **(gpu_kw or {}))
    o_ref, s_ref = oracle_forward(inp, **(oracle_kw or {}))
    o64 = o.double().cpu().numpy()
    s64 = s.double().cpu().numpy()
    assert np.all(np.isfinite(o64)) and np.all(np.isfinite(s64))
    out = (rel(o64, o_ref), rel(s64, s_ref), o, s)
    if units:
        cu = inp.get("cu_seqlens")
        cu = None if cu is None else cu.tolist()
        out = out + (worst_unit_o(o64, o_ref, cu), worst_unit_state(s64, s_ref))
    return out
