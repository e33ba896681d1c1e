"""CPU tests: the backward oracle against central finite differences of the
independent C oracle's forward, the beta = 0 closed form, and planted
mistakes that some pin must catch."""
import importlib.util

import numpy as np
import pytest

import oracle
import oracle.grad as OG
from pins import rel

SRC = OG.__file__


def _inputs(rng, B, T, H, dk, dv):
    q = rng.standard_normal((B, T, H, dk)) / np.sqrt(dk)
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    h0 = rng.standard_normal((B, H, dk, dv)) * 0.3
    return q, k, v, g, beta, h0


def _loss_c(q, k, v, g, beta, h0, d_o, dhN, cu=None):
    """The scalar the backward differentiates, on the C oracle's forward."""
    o, sN = oracle.forward(q, k, v, g, beta, h0, cu, threads=1)
    return float(np.sum(o * d_o) + np.sum(sN * dhN))


def pin_finite_differences(mod, seed=31):
    oracle.build()
    rng = np.random.default_rng(seed)
    out = []
    for (B, T, H, dk, dv, varlen) in ((1, 6, 2, 3, 2, False), (2, 4, 1, 2, 3, False),
                                      (1, 9, 1, 3, 2, True)):
        x = list(_inputs(rng, B, T, H, dk, dv))
        cu = None
        if varlen:
            cu = np.array([0, 4, 9], dtype=np.int64)
            x[5] = rng.standard_normal((2, H, dk, dv)) * 0.3
        d_o = rng.standard_normal((B, T, H, dv))
        dhN = rng.standard_normal(x[5].shape)
        gr = mod.backward(*x, d_o, dhN, cu)
        eps = 1e-5
        for i, name in enumerate(["dq", "dk", "dv", "dg", "dbeta", "dh0"]):
            d = rng.standard_normal(x[i].shape)
            xp = [a.copy() for a in x]; xm = [a.copy() for a in x]
            xp[i] = x[i] + eps * d; xm[i] = x[i] - eps * d
            fd = (_loss_c(*xp, d_o, dhN, cu) - _loss_c(*xm, d_o, dhN, cu)) / (2 * eps)
            an = float(np.sum(gr[name] * d))
            out.append((f"fd {name} B{B}T{T}{' varlen' if varlen else ''}",
                        abs(fd - an) / max(1.0, abs(fd)), 1e-7))
    return out


def pin_beta_zero(mod, seed=32):
    """beta = 0: H_t = exp(G_t) H_0, o_t = exp(G_t) H_0^T q_t, so
    dq_t = exp(G_t) H_0 do_t, dH_0 = sum_t exp(G_t) q_t do_t^T + exp(G_T) dH_N,
    dv = dk = 0, dg_t = sum_{s >= t} <do_s, o_s> + exp(G_T) <dH_N, H_0>."""
    rng = np.random.default_rng(seed)
    B, T, H, dk, dv = 1, 7, 2, 3, 4
    q, k, v, g, _, h0 = _inputs(rng, B, T, H, dk, dv)
    beta = np.zeros((B, T, H))
    d_o = rng.standard_normal((B, T, H, dv))
    dhN = rng.standard_normal((B, H, dk, dv))
    gr = mod.backward(q, k, v, g, beta, h0, d_o, dhN)
    G = np.cumsum(g, axis=1)                                          # [B, T, H]
    eG = np.exp(G)
    dq = eG[..., None] * np.einsum("bhkv,bthv->bthk", h0, d_o)
    dh0 = np.einsum("bth,bthk,bthv->bhkv", eG, q, d_o) + eG[:, -1][..., None, None] * dhN
    o = eG[..., None] * np.einsum("bhkv,bthk->bthv", h0, q)
    per_t = np.sum(d_o * o, axis=-1)                                  # [B, T, H]
    tail = eG[:, -1] * np.sum(dhN * h0, axis=(-2, -1))                # [B, H]
    dg = np.cumsum(per_t[:, ::-1], axis=1)[:, ::-1] + tail[:, None, :]
    return [("beta0 dq", rel(gr["dq"], dq), 1e-13), ("beta0 dh0", rel(gr["dh0"], dh0), 1e-13),
            ("beta0 dv", float(np.abs(gr["dv"]).max()), 0.0),
            ("beta0 dk", float(np.abs(gr["dk"]).max()), 0.0),
            ("beta0 dg", rel(gr["dg"], dg), 1e-13)]


def _bad(res):
    return [(l, e, b) for l, e, b in res if not e <= b]


def test_finite_differences():
    bad = _bad(pin_finite_differences(OG))
    assert not bad, bad


def test_beta_zero_closed_form():
    bad = _bad(pin_beta_zero(OG))
    assert not bad, bad


def test_forward_agrees_with_c_oracle():
    rng = np.random.default_rng(33)
    x = _inputs(rng, 2, 11, 2, 4, 3)
    d_o = rng.standard_normal((2, 11, 2, 3))
    gr = OG.backward(*x, d_o, None)
    o, sN = oracle.forward(*x, threads=1)
    assert rel(gr["o"], o) <= 1e-14 and rel(gr["final_state"], sN) <= 1e-14


MUTANTS = [
    ("erase sign", "Hs - bt * kt[:, :, None]", "Hs + bt * kt[:, :, None]"),
    ("decay on the write too", "Hs = a * (Hs - bt * kt[:, :, None] * kH[:, None, :]) + bt",
     "Hs = a * (Hs - bt * kt[:, :, None] * kH[:, None, :]) + a * bt"),
    ("read with the write key", "o_rows[row][t] = torch.einsum(\"hkv,hk->hv\", Hs, qt)",
     "o_rows[row][t] = torch.einsum(\"hkv,hk->hv\", Hs, kt)"),
    ("final-state gradient dropped", "loss = loss + (hN * dhN).sum()", "loss = loss"),
    ("decay exp sign", "a = torch.exp(g[row, t])", "a = torch.exp(-g[row, t])"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    path = tmp_path / "grad_mutant.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("grad_mutant", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    bad = _bad(pin_finite_differences(mod)) + _bad(pin_beta_zero(mod))
    assert bad, f"no pin caught the planted mistake: {name}"


def test_chunked_backward_equals_autograd():
    """The chunked (WY-form) statement of the backward, oracle.chunked_grad,
    equals the autograd oracle to fp64 rounding: several chunks, a ragged
    last chunk, packed sequences with an empty one, slow and fast gates."""
    import torch
    import oracle.chunked_grad as CG
    rng = np.random.default_rng(71)
    cases = [(1, 150, 2, 8, 4, None, 1.0), (2, 64, 1, 4, 6, None, 1.0),
             (1, 140, 1, 6, 5, [0, 70, 70, 71, 140], 0.01)]
    for B, T, H, dk, dv, cu, scale in cases:
        q, k, v, g, beta, _ = _inputs(rng, B, T, H, dk, dv)
        g = g * scale
        N = B if cu is None else len(cu) - 1
        h0 = rng.standard_normal((N, H, dk, dv)) * 0.3
        d_o = rng.standard_normal((B, T, H, dv))
        dhN = rng.standard_normal((N, H, dk, dv))
        t = [torch.from_numpy(x) for x in (q, k, v, g, beta, h0, d_o, dhN)]
        cu_t = None if cu is None else torch.tensor(cu)
        ref = OG.backward(t[0], t[1], t[2], t[3], t[4], t[5], t[6], t[7], cu_t)
        got = CG.backward(q, k, v, g, beta, h0, d_o, dhN, cu)
        for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
            assert rel(got[name], ref[name]) < 1e-10, (name, B, T, cu)
