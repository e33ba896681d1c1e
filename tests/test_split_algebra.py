"""CPU checks of the algebra the sequence split rests on, in fp64 with the
oracles alone: a run of tokens maps its entry state H to M H + X and each of
its outputs to o0 + r^T H, where X and o0 are the run from a zero state and M
and r the run from the identity with zero values.  Composing the segments'
maps and correcting their outputs must give the whole sequence's result (the
gated delta rule, and the diagonal decay combined with the delta rule)."""
from __future__ import annotations

import numpy as np

import oracle
import oracle.diag
from pins import rel


def _gdn_inputs(rng, T, H, dk, dv, gate_scale, beta_scale=0.1):
    q = rng.standard_normal((1, T, H, dk))
    k = rng.standard_normal((1, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, H, dv))
    g = -gate_scale * np.log1p(np.exp(rng.standard_normal((1, T, H))))
    beta = beta_scale / (1.0 + np.exp(-rng.standard_normal((1, T, H))))
    h0 = 0.5 * rng.standard_normal((1, H, dk, dv))
    return q, k, v, g, beta, h0


def test_gated_delta_rule_segments_compose():
    oracle.build()
    rng = np.random.default_rng(41)
    T, H, dk, dv = 150, 2, 8, 6
    q, k, v, g, beta, h0 = _gdn_inputs(rng, T, H, dk, dv, gate_scale=0.05)
    o_ref, s_ref = oracle.forward(q, k, v, g, beta, h0)
    cuts = [0, 40, 97, T]   # three segments, none aligned to anything
    eye = np.broadcast_to(np.eye(dk), (1, H, dk, dk)).copy()
    state = h0
    o = np.zeros_like(o_ref)
    for a, b in zip(cuts[:-1], cuts[1:]):
        seg = (q[:, a:b], k[:, a:b])
        o0, X = oracle.forward(*seg, v[:, a:b], g[:, a:b], beta[:, a:b], None)
        r, M = oracle.forward(*seg, np.zeros((1, b - a, H, dk)), g[:, a:b], beta[:, a:b], eye)
        # o_t = o0_t + r_t^T H (r_t has one entry per key row), H' = M H + X
        corr = np.einsum("bthk,bhkd->bthd", r, state)
        assert np.linalg.norm(corr) > 0.05 * np.linalg.norm(o0)   # the entry state carries weight
        o[:, a:b] = o0 + corr
        state = np.einsum("bhik,bhkd->bhid", M, state) + X
    assert rel(o, o_ref) < 1e-12
    assert rel(state, s_ref) < 1e-12


def test_gated_delta_rule_segment_map_is_not_trivial():
    """With slow gates a segment's M keeps weight (so the check above tests
    the composition, not a state that was forgotten)."""
    oracle.build()
    rng = np.random.default_rng(42)
    T, H, dk = 60, 1, 8
    q, k, _, g, beta, _ = _gdn_inputs(rng, T, H, dk, 4, gate_scale=0.05)
    eye = np.broadcast_to(np.eye(dk), (1, H, dk, dk)).copy()
    _, M = oracle.forward(q, k, np.zeros((1, T, H, dk)), g, beta, eye)
    assert np.linalg.norm(M) > 0.1


def test_diag_delta_segments_compose():
    rng = np.random.default_rng(43)
    B, T, H, S, D = 1, 90, 2, 6, 5
    v = rng.standard_normal((B, T, H, D))
    b = rng.standard_normal((B, T, H, S))
    b /= np.linalg.norm(b, axis=-1, keepdims=True)
    c = rng.standard_normal((B, T, H, S))
    g = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    A_log = rng.uniform(-4.0, -2.0, (H, S))   # slow, different per row
    beta = 0.1 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    h0 = rng.standard_normal((B, H, S, D))
    o_ref, s_ref = oracle.diag.forward_delta(v, b, c, g, A_log, beta, h0)
    cuts = [0, 33, 61, T]
    eye = np.broadcast_to(np.eye(S), (B, H, S, S)).copy()
    state = h0
    o = np.zeros_like(o_ref)
    for a, e in zip(cuts[:-1], cuts[1:]):
        sl = slice(a, e)
        o0, X = oracle.diag.forward_delta(v[:, sl], b[:, sl], c[:, sl], g[:, sl], A_log,
                                          beta[:, sl], None)
        r, M = oracle.diag.forward_delta(np.zeros((B, e - a, H, S)), b[:, sl], c[:, sl],
                                         g[:, sl], A_log, beta[:, sl], eye)
        corr = np.einsum("bths,bhsd->bthd", r, state)
        assert np.linalg.norm(corr) > 0.05 * np.linalg.norm(o0)   # the entry state carries weight
        o[:, sl] = o0 + corr
        state = np.einsum("bhis,bhsd->bhid", M, state) + X
    assert rel(o, o_ref) < 1e-12
    assert rel(state, s_ref) < 1e-12
