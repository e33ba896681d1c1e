"""CPU tests: the oracle against the pins that the mathematics fixes.

Each test prints nothing on success; on failure it lists every violated bound.
"""
import functools

import numpy as np
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def fwd():
    oracle.build()
    return oracle.forward


def _check(results):
    bad = pins.run(results)
    assert not bad, "pin violated: " + "; ".join(f"{l}: {e:.3e} > {b:.0e}" for l, e, b in bad)


def test_golden_two_token(fwd):
    _check(pins.pin_golden_two_token(fwd))


def test_p1_beta_zero_closed_form(fwd):
    _check(pins.pin_beta_zero_closed_form(fwd))


def test_p2_gla_closed_form(fwd):
    _check(pins.pin_gla_closed_form(functools.partial(fwd, mode=oracle.MODE_GLA)))


def test_p3_exact_overwrite(fwd):
    _check(pins.pin_exact_overwrite(fwd))


def test_p4_chunked_equals_sequential(fwd):
    _check(pins.pin_chunked_equals_sequential(fwd, oracle.chunked.forward))


def test_p5_state_chaining(fwd):
    _check(pins.pin_state_chaining(fwd))


def test_p6_exact_brute_force(fwd):
    _check(pins.pin_brute_force(fwd))


def test_p7_nonexpansive(fwd):
    _check(pins.pin_nonexpansive(fwd))


def test_p7_varlen_bitwise(fwd):
    _check(pins.pin_varlen_bitwise(fwd))


def test_thread_count_does_not_change_result(fwd):
    rng = np.random.default_rng(11)
    q, k, v, g, beta = pins._inputs(rng, 3, 50, 4, 8, 8)
    o1, s1 = fwd(q, k, v, g, beta, threads=1)
    o8, s8 = fwd(q, k, v, g, beta, threads=8)
    assert np.array_equal(o1, o8) and np.array_equal(s1, s8)


def test_qk_l2norm_option(fwd):
    """The optional q/k normalisation: x / sqrt(|x|^2 + 1e-6).

    Pinned by (a) invariance to positive per-row rescaling of q and k (exact up
    to the 1e-6 epsilon), and (b) near-identity on rows that already have unit
    norm (a factor 1/sqrt(1 + 1e-6) per row)."""
    rng = np.random.default_rng(12)
    B, T, H, dk, dv = 1, 70, 2, 8, 6
    q, k, v, g, beta = pins._inputs(rng, B, T, H, dk, dv)
    cq = rng.uniform(2.0, 30.0, (B, T, H, 1))
    ck = rng.uniform(2.0, 30.0, (B, T, H, 1))
    o_ref, s_ref = fwd(q, k, v, g, beta)
    o_n, s_n = fwd(q * cq, k * ck, v, g, beta, qk_l2norm=True)
    assert pins.rel(o_n, o_ref) < 1e-5 and pins.rel(s_n, s_ref) < 1e-5
    o_u, s_u = fwd(q, k, v, g, beta, qk_l2norm=True)
    assert pins.rel(o_u, o_ref) < 3e-6 and pins.rel(s_u, s_ref) < 3e-6
    # without the option the rescaled inputs give a different answer
    o_raw, _ = fwd(q * cq, k * ck, v, g, beta)
    assert pins.rel(o_raw, o_ref) > 1e-2


def test_final_state_optional_and_zero_length(fwd):
    rng = np.random.default_rng(13)
    q, k, v, g, beta = pins._inputs(rng, 1, 20, 1, 4, 4)
    H0 = rng.standard_normal((3, 1, 4, 4))
    cu = np.array([0, 0, 20, 20])
    o, s = fwd(q, k, v, g, beta, H0, cu)
    # an empty sequence hands its initial state through unchanged
    assert np.array_equal(s[0], H0[0]) and np.array_equal(s[2], H0[2])
    o2, s2 = fwd(q, k, v, g, beta, H0, cu, return_final_state=False)
    assert s2 is None and np.array_equal(o, o2)
