"""GPU parity of ``gdn_diag_delta_fwd`` (the pages' diagonal decay combined
with the delta rule) against the fp64 oracle ``oracle.diag.forward_delta`` on
the same seeded inputs, through the C ABI."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle.block as OB
import oracle.diag
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W
from parity import MARGINS, TOL, rel, worst_unit_state

pytestmark = pytest.mark.gpu


def _dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _gpu(d, **kw):
    x = _dev(d)
    o, s = G.gdn_diag_delta_fwd(x["v"], x["b"], x["c"], x["g"], x["A_log"], x["beta"],
                                x["initial_state"], check=True, **kw)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), s.double().cpu().numpy()


def _oracle(d, g=None, beta=None):
    return oracle.diag.forward_delta(d["v"], d["b"], d["c"], d["g"] if g is None else g,
                                     d["A_log"], d["beta"] if beta is None else beta,
                                     d["initial_state"])


def _case(dtype, B, T, H, a_log, init, seed):
    return W.generate_diag(W.DiagWorkload("t", B=B, T=T, H=H, dtype=dtype, a_log=a_log,
                                          init_state=init, delta=True, seed=seed))


def _tol(dtype):
    return TOL[W._DTYPES[dtype]]


# one token, a partial tile, whole tiles, one and several 128-token segments
# with ragged tails
SIZES = [(1, 1, 1), (1, 15, 2), (1, 16, 1), (2, 17, 2), (1, 128, 1), (1, 129, 2),
         (2, 300, 3), (1, 1000, 2)]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,H", SIZES, ids=[f"B{b}T{t}H{h}" for b, t, h in SIZES])
@pytest.mark.parametrize("init", [False, True])
def test_diag_delta_matches_oracle(dtype, B, T, H, init):
    d = _case(dtype, B, T, H, "uniform", init, B * 1000 + T + H)
    o, s = _gpu(d)
    o_ref, s_ref = _oracle(d)
    to, ts = _tol(dtype)
    assert rel(o, o_ref) <= to
    assert rel(s, s_ref) <= ts
    assert worst_unit_state(s, s_ref) <= ts


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("a_log,T,H", [("pages", 300, 40), ("slow", 2000, 4),
                                       ("slow", 4097, 2)])
def test_diag_delta_decay_regimes(dtype, a_log, T, H):
    """The pages' initialisation (A = -1 .. -40: most heads forget within a
    token) and slow decays (the state carried through every segment's map,
    many segments deep)."""
    d = _case(dtype, 2, T, H, a_log, True, 7)
    o, s = _gpu(d)
    o_ref, s_ref = _oracle(d)
    to, ts = _tol(dtype)
    assert rel(o, o_ref) <= to
    assert rel(s, s_ref) <= ts
    assert worst_unit_state(s, s_ref) <= ts


def test_diag_delta_overwrite():
    """beta = 1, unit write keys and c = b: every output is v (the delta
    rule's overwrite), across segment boundaries and with an initial state."""
    d = _case("fp32", 2, 400, 3, "uniform", True, 11)
    d["beta"] = torch.ones_like(d["beta"])
    d["c"] = d["b"].clone()
    o, _ = _gpu(d)
    assert rel(o, d["v"].double().numpy()) <= 1e-4


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("parts", ["all", "skip", "gate", "sigmoids"])
def test_diag_delta_block_parts(dtype, parts):
    """The gate and beta as logits (sigmoid in the kernel) and the block
    epilogue (o + D v) * gate, against the oracle composed with the
    epilogue's oracle."""
    B, T, H = 2, 333, 3
    d = _case(dtype, B, T, H, "uniform", True, 21)
    rng = np.random.default_rng(22)
    dt = torch.from_numpy(rng.standard_normal((B, T, H))).to(torch.float32)
    blog = torch.from_numpy(rng.standard_normal((B, T, H))).to(d["v"].dtype)
    D_skip = torch.from_numpy(rng.standard_normal(H)).to(torch.float32)
    gate = torch.from_numpy(OB.sigmoid(rng.standard_normal((B, T, H)))).to(torch.float32)
    skip, gt, sig = parts in ("all", "skip"), parts in ("all", "gate"), parts in ("all", "sigmoids")
    x = _dev(d)
    o, s = G.gdn_diag_delta_fwd(x["v"], x["b"], x["c"], dt.cuda() if sig else x["g"],
                                x["A_log"], blog.cuda() if sig else x["beta"],
                                x["initial_state"], D_skip=D_skip.cuda() if skip else None,
                                out_gate=gate.cuda() if gt else None, gate_sigmoid=sig,
                                beta_logits=sig, check=True)
    torch.cuda.synchronize()
    o_rec, s_ref = _oracle(d, g=OB.sigmoid(dt) if sig else None,
                           beta=OB.sigmoid(blog.double()) if sig else None)
    o_ref = OB.epilogue(o_rec, d["v"], D_skip if skip else np.zeros(H),
                        gate if gt else np.ones((B, T, H)))
    to, ts = _tol(dtype)
    assert rel(o.double().cpu().numpy(), o_ref) <= to
    assert rel(s.double().cpu().numpy(), s_ref) <= ts


def test_diag_delta_workspace_reused_across_calls():
    """One workspace across calls: the launch counter and the flags' epoch
    tag advance each call, so no call reads an end state of an earlier one."""
    d = _case("fp32", 2, 700, 3, "slow", True, 3)
    x = _dev(d)
    ws = G.new_diag_delta_workspace(2, 700, 3, 32, 32)
    o_ref, s_ref = _oracle(d)
    for i in range(4):
        v = x["v"] if i % 2 == 0 else -x["v"]   # odd calls: every result negated
        o, s = G.gdn_diag_delta_fwd(v, x["b"], x["c"], x["g"], x["A_log"], x["beta"],
                                    x["initial_state"] if i % 2 == 0 else -x["initial_state"],
                                    workspace=ws, check=True)
        torch.cuda.synchronize()
        sign = 1.0 if i % 2 == 0 else -1.0
        assert rel(o.double().cpu().numpy(), sign * o_ref) <= 1e-4
        assert rel(s.double().cpu().numpy(), sign * s_ref) <= 1e-4


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_diag_delta_chaining(dtype):
    """Two calls chained through the state against the oracle over the whole
    sequence (the cut inside a segment)."""
    d = _case(dtype, 2, 500, 2, "slow", True, 5)
    m = 211
    cut = ("v", "b", "c", "g", "beta")
    first = {k: (v[:, :m].contiguous() if k in cut else v) for k, v in d.items()}
    o1, s1 = _gpu(first)
    second = {k: (v[:, m:].contiguous() if k in cut else v) for k, v in d.items()}
    second["initial_state"] = torch.from_numpy(s1).float()
    o2, s2 = _gpu(second)
    o_ref, s_ref = _oracle(d)
    to, ts = _tol(dtype)
    assert rel(np.concatenate([o1, o2], axis=1), o_ref) <= to
    assert rel(s2, s_ref) <= ts


def test_diag_delta_full_size_sampled():
    """The pages' production shape with the erase added (B=4, T=4096, H=40,
    bf16) in the launch configuration the benchmark times; the oracle runs on
    sampled heads, a slow-decay copy of it on the same heads."""
    w = W.DIAG_WORKLOADS["hymo_diag_delta_bf16"]
    to, ts = _tol("bf16")
    for wl in (w, dataclasses.replace(w, a_log="slow", seed=1)):
        d = W.generate_diag(wl)
        o, s = _gpu(d)
        worst = 0.0
        for (b, h) in [(0, 0), (1, 7), (3, 39), (2, 20)]:
            sub = {k: d[k][b:b + 1, :, h:h + 1] for k in ("v", "b", "c", "g", "beta")}
            sub["A_log"] = d["A_log"][h:h + 1]
            sub["initial_state"] = None
            o_ref, s_ref = _oracle(sub)
            eo, es = rel(o[b:b + 1, :, h:h + 1], o_ref), rel(s[b:b + 1, h:h + 1], s_ref)
            worst = max(worst, eo)
            assert eo <= to and es <= ts, (wl.a_log, b, h)
        MARGINS.append(f"{wl.name} (A_log {wl.a_log}) [diag_delta]: worst sampled head "
                       f"o={worst:.3e}")
