"""CPU tests: the block prologue/epilogue oracle against PyTorch's own CPU
conv1d and SiLU (library routines), impulse responses, chaining, a worked
example, and planted mistakes that some pin must catch."""
import importlib.util
import json
import os

import numpy as np
import pytest
import torch

import oracle.block as OB
from pins import GOLDEN, rel

SRC = OB.__file__


def _torch_conv_silu(x, w, x_prev=None):
    """PyTorch's depthwise Conv1d (groups = C, padding K-1, tail trimmed) and SiLU, fp64."""
    B, T, C = x.shape
    K = w.shape[1]
    xt = torch.from_numpy(x).permute(0, 2, 1)                          # [B, C, T]
    if x_prev is not None:
        xt = torch.cat([torch.from_numpy(x_prev).permute(0, 2, 1), xt], dim=2)
        z = torch.nn.functional.conv1d(xt, torch.from_numpy(w)[:, None, :], groups=C)
    else:
        z = torch.nn.functional.conv1d(xt, torch.from_numpy(w)[:, None, :], groups=C,
                                       padding=K - 1)[..., :T]
    return torch.nn.functional.silu(z).permute(0, 2, 1).numpy()


def pins(mod):
    rng = np.random.default_rng(21)
    out = []
    for (B, T, C, K) in ((2, 37, 6, 4), (1, 9, 3, 2), (3, 5, 4, 3), (1, 2, 5, 4)):
        x = rng.standard_normal((B, T, C))
        w = rng.standard_normal((C, K))
        y, _ = mod.conv_silu(x, w)
        out.append((f"torch conv1d+silu K={K}", rel(y, _torch_conv_silu(x, w)), 1e-13))
        xp = rng.standard_normal((B, K - 1, C))
        y, _ = mod.conv_silu(x, w, xp)
        out.append((f"torch conv1d+silu prefix K={K}", rel(y, _torch_conv_silu(x, w, xp)), 1e-13))
    # impulse: a unit input at token s gives pre-activations w[:, K-1], ..., w[:, 0] at s, s+1, ...
    B, T, C, K = 1, 12, 3, 4
    w = rng.standard_normal((C, K))
    x = np.zeros((B, T, C))
    s = 5
    x[0, s, :] = 1.0
    y, _ = mod.conv_silu(x, w)
    z = np.zeros((T, C))
    for d in range(K):
        z[s + d] = w[:, K - 1 - d]
    out.append(("impulse response", rel(y[0], z / (1.0 + np.exp(-z))), 1e-14))
    # chaining: two calls through the tail equal one call
    x = rng.standard_normal((2, 30, 4))
    w = rng.standard_normal((4, 4))
    y, tail = mod.conv_silu(x, w)
    y1, t1 = mod.conv_silu(x[:, :13], w)
    y2, t2 = mod.conv_silu(x[:, 13:], w, t1)
    out.append(("chained y", rel(np.concatenate([y1, y2], axis=1), y), 1e-15))
    out.append(("chained tail", rel(t2, tail), 0.0))
    # a call shorter than the window: the tail mixes prefix and input
    xp = rng.standard_normal((2, 3, 4))
    _, t = mod.conv_silu(x[:, :2], w, xp)
    out.append(("short tail", rel(t, np.concatenate([xp[:, 2:], x[:, :2]], axis=1)), 0.0))
    # epilogue: the hand-worked example
    with open(os.path.join(GOLDEN, "block_epilogue_hand.json")) as f:
        gold = json.load(f)
    o = np.array(gold["o"])[None, None]
    v = np.array(gold["v"])[None, None]
    e = mod.epilogue(o, v, np.array(gold["D"]), np.array(gold["g_gate"])[None, None])
    out.append(("epilogue golden", rel(e[0, 0], gold["out"]), 1e-15))
    out.append(("sigmoid(0) = 1/2", abs(float(mod.sigmoid(0.0)) - 0.5), 0.0))
    out.append(("sigmoid(log 3) = 3/4", abs(float(mod.sigmoid(np.log(3.0))) - 0.75), 1e-15))
    return out


def _bad(results):
    return [(l, e, b) for l, e, b in results if not e <= b]


def test_block_oracle_pins():
    bad = _bad(pins(OB))
    assert not bad, bad


MUTANTS = [
    ("taps reversed", "w[None, None, :, k] * xs[:, k:k + T, :]",
     "w[None, None, :, K - 1 - k] * xs[:, k:k + T, :]"),
    ("not causal (centred)", "xs[:, k:k + T, :]", "xs[:, min(k + 1, K - 1):min(k + 1, K - 1) + T, :]"),
    ("silu dropped", "y = z * sigmoid(z)", "y = z"),
    ("sigmoid instead of silu", "y = z * sigmoid(z)", "y = sigmoid(z)"),
    ("prefix ignored", "prev = np.zeros((B, K - 1, C)) if x_prev is None else _f64(x_prev)",
     "prev = np.zeros((B, K - 1, C))"),
    ("skip after the gate", "(o + D[None, None, :, None] * v) * g_gate[..., None]",
     "o * g_gate[..., None] + D[None, None, :, None] * v"),
    ("gate sign", "1.0 / (1.0 + np.exp(-z))", "1.0 / (1.0 + np.exp(z))"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    path = tmp_path / "block_mutant.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("block_mutant", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    try:
        failing = _bad(pins(mod))
    except (ValueError, IndexError):
        failing = ["shape error"]
    assert failing, f"no pin caught the planted mistake: {name}"
