"""CPU tests: the diagonal-decay oracle against its pins, and planted mistakes
in copies of the oracle's source that some pin must catch."""
import functools
import importlib.util
import os

import pytest

import oracle
import oracle.diag
import pins
import pins_diag

SRC = oracle.diag.__file__


def _gla():
    oracle.build()
    return functools.partial(oracle.forward, mode=oracle.MODE_GLA)


def _check(results):
    bad = pins.run(results)
    assert not bad, "pin violated: " + "; ".join(f"{l}: {e:.3e} > {b:.0e}" for l, e, b in bad)


def test_golden_page_decay():
    _check(pins_diag.pin_golden_page_decay(oracle.diag.forward))


def test_unrolled_closed_form():
    _check(pins_diag.pin_unrolled(oracle.diag.forward))


def test_linear_attention_limit():
    _check(pins_diag.pin_linear_attention(oracle.diag.forward))


def test_scalar_decay_equals_sequential_oracle():
    _check(pins_diag.pin_scalar_decay(oracle.diag.forward, _gla()))


def test_row_independence():
    _check(pins_diag.pin_row_independence(oracle.diag.forward))


def test_chaining():
    _check(pins_diag.pin_chaining(oracle.diag.forward))


def _gdn():
    oracle.build()
    return oracle.forward


def test_delta_scalar_rates_equal_gated_delta_rule():
    _check(pins_diag.pin_delta_scalar_rates(oracle.diag.forward_delta, _gdn()))


def test_delta_pure_decay():
    _check(pins_diag.pin_delta_pure_decay(oracle.diag.forward_delta))


def test_delta_overwrite():
    _check(pins_diag.pin_delta_overwrite(oracle.diag.forward_delta))


def test_delta_basis_keys():
    _check(pins_diag.pin_delta_basis_keys(oracle.diag.forward_delta))


def test_delta_chaining():
    _check(pins_diag.pin_delta_chaining(oracle.diag.forward_delta))


# (name, text in oracle/diag.py, replacement)
MUTANTS = [
    ("decay grows (A sign)", "A = -np.exp(A_log)", "A = np.exp(A_log)"),
    ("decay ignores the gate", "np.exp(g[:, t, :, None] * A[None, :, :])",
     "np.exp(A[None, :, :] + 0 * g[:, t, :, None])"),
    ("decay per value column", "decay[..., None] * h", "decay[..., None, :] * h"),
    ("read before write", "o[:, t] = np.einsum(\"bhs,bhsd->bhd\", c[:, t], h)\n",
     "pass\n"),
    ("decay applied after the write",
     "h = decay[..., None] * h + b[:, t, :, :, None] * v[:, t, :, None, :]",
     "h = decay[..., None] * (h + b[:, t, :, :, None] * v[:, t, :, None, :])"),
    ("read with the write key", "c[:, t], h)", "b[:, t], h)"),
    ("gate of the next token", "g[:, t, :, None]", "g[:, min(t + 1, g.shape[1] - 1), :, None]"),
    ("initial state dropped", "else _f64(initial_state).copy()", "else 0 * _f64(initial_state)"),
]


def _load_mutant(path):
    spec = importlib.util.spec_from_file_location("diag_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    if name == "read before write":
        # read the state before the update: move the read above the write
        mutated = mutated.replace(
            "        h = decay[..., None] * h",
            "        o[:, t] = np.einsum(\"bhs,bhsd->bhd\", c[:, t], h)\n"
            "        h = decay[..., None] * h", 1)
    path = tmp_path / "diag_mutant.py"
    path.write_text(mutated)
    mod = _load_mutant(str(path))
    try:
        failing = pins.run(pins_diag.all_pins(mod.forward, _gla()))
    except (ValueError, IndexError):
        failing = ["shape error"]          # a mutant that cannot even run is caught
    assert failing, f"no pin caught the planted mistake: {name}"


# Planted mistakes in forward_delta (anchors that occur only there).
MUTANTS_DELTA = [
    ("erase reads the undecayed state", 'pred = np.einsum("bhs,bhsd->bhd", bt, hbar)',
     'pred = np.einsum("bhs,bhsd->bhd", bt, h)'),
    ("write without beta", "err = beta[:, t, :, None] * (v[:, t] - pred)",
     "err = (v[:, t] - pred)"),
    ("erase without beta", "err = beta[:, t, :, None] * (v[:, t] - pred)",
     "err = beta[:, t, :, None] * v[:, t] - pred"),
    ("decay after the update", "h = hbar + bt[..., None] * err[:, :, None, :]",
     "h = decay[..., None] * (h + bt[..., None] * err[:, :, None, :])"),
    ("delta decay per value column", "hbar = decay[..., None] * h",
     "hbar = decay[..., None, :] * h"),
    ("erase sign", "h = hbar + bt[..., None] * err[:, :, None, :]",
     "h = hbar - bt[..., None] * err[:, :, None, :]"),
    ("delta read with the write key",
     'err[:, :, None, :]\n        o[:, t] = np.einsum("bhs,bhsd->bhd", c[:, t], h)',
     'err[:, :, None, :]\n        o[:, t] = np.einsum("bhs,bhsd->bhd", bt, h)'),
]


@pytest.mark.parametrize("name,old,new", MUTANTS_DELTA, ids=[m[0] for m in MUTANTS_DELTA])
def test_delta_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    path = tmp_path / "diag_delta_mutant.py"
    path.write_text(src.replace(old, new, 1))
    mod = _load_mutant(str(path))
    try:
        failing = pins.run(pins_diag.all_delta_pins(mod.forward_delta, _gdn()))
    except (ValueError, IndexError):
        failing = ["shape error"]
    assert failing, f"no pin caught the planted mistake: {name}"
