"""GPU parity of ``gdn_diag_fwd`` (the pages' diagonal-decay recurrence)
against the fp64 oracle ``oracle.diag`` on the same seeded inputs, through
the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.diag
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W
from parity import TOL, rel

pytestmark = pytest.mark.gpu


def _dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _gpu(d, **kw):
    x = _dev(d)
    o, s = G.gdn_diag_fwd(x["v"], x["b"], x["c"], x["g"], x["A_log"], x["initial_state"],
                          check=True, **kw)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), s.double().cpu().numpy()


def _oracle(d):
    return oracle.diag.forward(d["v"], d["b"], d["c"], d["g"], d["A_log"], d["initial_state"])


def _tol(dtype):
    return TOL[W._DTYPES[dtype]]


SIZES = [(1, 1, 1), (1, 15, 2), (1, 16, 1), (2, 17, 2), (1, 128, 1), (1, 129, 2),
         (2, 300, 3), (1, 1000, 2)]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,H", SIZES, ids=[f"B{b}T{t}H{h}" for b, t, h in SIZES])
@pytest.mark.parametrize("init", [False, True])
def test_diag_matches_oracle(dtype, B, T, H, init):
    w = W.DiagWorkload("t", B=B, T=T, H=H, dtype=dtype, a_log="uniform", init_state=init,
                       seed=B * 1000 + T + H)
    d = W.generate_diag(w)
    o, s = _gpu(d)
    o_ref, s_ref = _oracle(d)
    to, ts = _tol(dtype)
    assert rel(o, o_ref) <= to
    assert rel(s, s_ref) <= ts


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("a_log,T", [("pages", 300), ("slow", 2000)])
def test_diag_decay_regimes(dtype, a_log, T):
    """The pages' initialisation (A = -1 .. -40: most heads forget within a
    token, products underflow) and slow decays (state carried across many
    128-token blocks, through the look-back)."""
    w = W.DiagWorkload("t", B=2, T=T, H=40 if a_log == "pages" else 4, dtype=dtype,
                       a_log=a_log, init_state=True, seed=7)
    d = W.generate_diag(w)
    o, s = _gpu(d)
    o_ref, s_ref = _oracle(d)
    to, ts = _tol(dtype)
    assert rel(o, o_ref) <= to
    assert rel(s, s_ref) <= ts


def test_diag_workspace_reused_across_calls():
    """One workspace across calls (its launch counter advances each call)."""
    w = W.DiagWorkload("t", B=2, T=700, H=3, dtype="fp32", a_log="slow", init_state=True,
                       seed=3)
    d = W.generate_diag(w)
    x = _dev(d)
    ws = G.new_diag_workspace(2, 700, 3, 32, 32)
    o_ref, s_ref = _oracle(d)
    for _ in range(4):
        o, s = G.gdn_diag_fwd(x["v"], x["b"], x["c"], x["g"], x["A_log"], x["initial_state"],
                              workspace=ws, check=True)
        torch.cuda.synchronize()
        assert rel(o.double().cpu().numpy(), o_ref) <= 1e-4
        assert rel(s.double().cpu().numpy(), s_ref) <= 1e-4


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_diag_chaining(dtype):
    """Two calls chained through the state (final_state into initial_state)
    against the oracle over the whole sequence."""
    w = W.DiagWorkload("t", B=2, T=500, H=2, dtype=dtype, a_log="slow", init_state=True,
                       seed=5)
    d = W.generate_diag(w)
    m = 211
    first = {k: (v[:, :m].contiguous() if k in ("v", "b", "c", "g") else v)
             for k, v in d.items()}
    o1, s1 = _gpu(first)
    second = {k: (v[:, m:].contiguous() if k in ("v", "b", "c", "g") else v)
              for k, v in d.items()}
    second["initial_state"] = torch.from_numpy(s1).float()
    o2, s2 = _gpu(second)
    o_ref, s_ref = _oracle(d)
    to, ts = _tol(dtype)
    assert rel(np.concatenate([o1, o2], axis=1), o_ref) <= to
    assert rel(s2, s_ref) <= ts


def test_diag_zero_values():
    """v = 0: with no initial state every output and the final state are
    exactly 0; with one, the outputs read the decayed initial state."""
    w = W.DiagWorkload("t", B=1, T=260, H=2, dtype="fp32", a_log="slow", init_state=True,
                       seed=9)
    d = W.generate_diag(w)
    d["v"] = torch.zeros_like(d["v"])
    o, s = _gpu(d)
    o_ref, s_ref = _oracle(d)
    assert rel(o, o_ref) <= 1e-4
    assert rel(s, s_ref) <= 1e-4
    d["initial_state"] = None
    o, s = _gpu(d)
    assert not np.any(o) and not np.any(s)


def test_diag_full_size_sampled():
    """The pages' production layer (B=4, T=4096, H=40, bf16) in the launch
    configuration the benchmark times; the oracle runs on sampled heads."""
    w = W.DIAG_WORKLOADS["hymo_diag_bf16"]
    d = W.generate_diag(w)
    o, s = _gpu(d)
    to, ts = _tol("bf16")
    for (b, h) in [(0, 0), (1, 7), (3, 39), (2, 20)]:
        sub = {"v": d["v"][b:b + 1, :, h:h + 1], "b": d["b"][b:b + 1, :, h:h + 1],
               "c": d["c"][b:b + 1, :, h:h + 1], "g": d["g"][b:b + 1, :, h:h + 1],
               "A_log": d["A_log"][h:h + 1], "initial_state": None}
        o_ref, s_ref = _oracle(sub)
        assert rel(o[b:b + 1, :, h:h + 1], o_ref) <= to, (b, h)
        assert rel(s[b:b + 1, h:h + 1], s_ref) <= ts, (b, h)
