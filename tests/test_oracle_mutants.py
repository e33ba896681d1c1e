"""CPU tests: plant plausible mistakes in a copy of the oracle's C source and
check that at least one pin catches each.  The copies are built under a
temporary directory; the oracle's own source and build are untouched."""
import ctypes
import functools
import os
import subprocess

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("erase sign flipped", "*s - beta * Sk[j] * k[i]", "*s + beta * Sk[j] * k[i]"),
    ("beta dropped from the write", "+ beta * v[j] * k[i]", "+ v[j] * k[i]"),
    ("decay applied to the erase only",
     "alpha * (*s - beta * Sk[j] * k[i])", "(*s - alpha * beta * Sk[j] * k[i])"),
    ("decay exponent sign", "exp(J->g[row])", "exp(-J->g[row])"),
    ("output read with the key", "acc += S[(size_t)j * dk + i] * q[i];",
     "acc += S[(size_t)j * dk + i] * k[i];"),
    ("erase projects the query", "acc += S[(size_t)j * dk + i] * k[i];\n        Sk[j]",
     "acc += S[(size_t)j * dk + i] * q[i];\n        Sk[j]"),
    ("final state stored untransposed",
     "= S[(size_t)j * dk + i];\n}", "= S[(size_t)i * dv + j];\n}"),
    ("initial state read transposed",
     "J->s0[state_off + (size_t)i * dv + j]", "J->s0[state_off + (size_t)j * dk + i]"),
    ("gate of the next token", "exp(J->g[row])",
     "exp(J->g[t + 1 < J->cu[n + 1] ? row + H : row])"),
]


def _all_pins(fwd):
    res = []
    res += pins.pin_golden_two_token(fwd)
    res += pins.pin_beta_zero_closed_form(fwd)
    res += pins.pin_gla_closed_form(functools.partial(fwd, mode=oracle.MODE_GLA))
    res += pins.pin_exact_overwrite(fwd)
    res += pins.pin_chunked_equals_sequential(fwd, oracle.chunked.forward)
    res += pins.pin_state_chaining(fwd)
    res += pins.pin_brute_force(fwd)
    return res


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path, monkeypatch):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-std=c11", "-o", str(so), str(c), "-lm"], check=True)
    lib = oracle._bind(ctypes.CDLL(str(so)))
    monkeypatch.setattr(oracle, "_lib", lib)
    failing = pins.run(_all_pins(oracle.forward))
    assert failing, f"no pin caught the planted mistake: {name}"
