"""GPU parity of the GDN block prologue (``gdn_conv_silu``) and of the block
epilogue and sigmoid gate fused into ``gdn_diag_fwd``, against the fp64
oracles ``oracle.block`` and ``oracle.diag``, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.block as OB
import oracle.diag as OD
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W
from parity import TOL, rel

pytestmark = pytest.mark.gpu

# conv + SiLU has no accumulation: fp32 output to fp32 rounding of a few
# operations; bf16 output to its own rounding (2^-9 relative) twice over.
CONV_TOL = {"fp32": 1e-5, "bf16": 4e-3}
DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


def _conv_inputs(B, T, C, K, dtype, seed, prefix):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((B, T, C))).to(DT[dtype])
    w = torch.from_numpy(rng.standard_normal((C, K)) * 0.5).to(torch.float32)
    xp = torch.from_numpy(rng.standard_normal((B, K - 1, C))).to(DT[dtype]) if prefix else None
    return x, w, xp


# C = 12 in bf16 (24-byte token rows) takes the kernel that loads through
# registers; every other case the TMA-staged one
CONV_CASES = [(1, 1, 8, 4), (2, 3, 16, 4), (1, 31, 40, 4), (2, 33, 1280, 4), (1, 257, 64, 3),
              (1, 100, 24, 2), (1, 50, 8, 1), (3, 600, 136, 4), (2, 130, 12, 4), (1, 70, 12, 3)]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,C,K", CONV_CASES, ids=[f"B{b}T{t}C{c}K{k}" for b, t, c, k in CONV_CASES])
@pytest.mark.parametrize("prefix", [False, True])
def test_conv_silu_matches_oracle(dtype, B, T, C, K, prefix):
    x, w, xp = _conv_inputs(B, T, C, K, dtype, B * 7 + T + C + K, prefix and K > 1)
    tail = torch.empty((B, K - 1, C), dtype=x.dtype, device="cuda") if K > 1 else None
    y = G.gdn_conv_silu(x.cuda(), w.cuda(), None if xp is None else xp.cuda(), x_tail=tail)
    torch.cuda.synchronize()
    y_ref, t_ref = OB.conv_silu(x, w, xp)
    assert rel(y.double().cpu().numpy(), y_ref) <= CONV_TOL[dtype]
    if tail is not None:
        assert np.array_equal(tail.double().cpu().numpy(), t_ref)   # a copy of inputs: exact


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_conv_silu_chained_calls_equal_one_call(dtype):
    """A sequence fed in three pieces through the prefix gives the one-call
    output bit for bit (each output is the same arithmetic on the same inputs)."""
    x, w, _ = _conv_inputs(2, 300, 128, 4, dtype, 3, False)
    xd, wd = x.cuda(), w.cuda()
    y = G.gdn_conv_silu(xd, wd)
    bufs = [torch.empty((2, 3, 128), dtype=x.dtype, device="cuda") for _ in range(2)]
    pieces, prev = [], None
    for i, (a, b) in enumerate(((0, 70), (70, 71), (71, 300))):
        pieces.append(G.gdn_conv_silu(xd[:, a:b].contiguous(), wd, prev, x_tail=bufs[i % 2]))
        prev = bufs[i % 2]
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(pieces, dim=1), y)


def test_conv_silu_full_size():
    """The pages' prologue shape: B=4, T=4096, d_inner=1280, d_conv=4, bf16."""
    x, w, _ = _conv_inputs(4, 4096, 1280, 4, "bf16", 11, False)
    y = G.gdn_conv_silu(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    y_ref, _ = OB.conv_silu(x, w)
    assert rel(y.double().cpu().numpy(), y_ref) <= CONV_TOL["bf16"]


def _diag_block_case(dtype, B, T, H, seed):
    w = W.DiagWorkload("t", B=B, T=T, H=H, dtype=dtype, a_log="uniform", init_state=True,
                       seed=seed)
    d = W.generate_diag(w)
    rng = np.random.default_rng(seed + 1)
    dt = torch.from_numpy(rng.standard_normal((B, T, H))).to(torch.float32)
    D_skip = torch.from_numpy(rng.standard_normal(H)).to(torch.float32)
    gate = torch.from_numpy(OB.sigmoid(rng.standard_normal((B, T, H)))).to(torch.float32)
    return d, dt, D_skip, gate


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,H", [(1, 1, 1), (2, 17, 2), (1, 300, 3), (2, 1000, 2)])
@pytest.mark.parametrize("parts", ["all", "skip", "gate", "sigmoid"])
def test_diag_block_epilogue_matches_oracle(dtype, B, T, H, parts):
    d, dt, D_skip, gate = _diag_block_case(dtype, B, T, H, B * 100 + T + H)
    use_skip = parts in ("all", "skip")
    use_gate = parts in ("all", "gate")
    use_sig = parts in ("all", "sigmoid")
    g_in = dt if use_sig else d["g"]
    x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    o, s = G.gdn_diag_fwd(x["v"], x["b"], x["c"], g_in.cuda(), x["A_log"], x["initial_state"],
                          D_skip=D_skip.cuda() if use_skip else None,
                          out_gate=gate.cuda() if use_gate else None,
                          gate_sigmoid=use_sig, check=True)
    torch.cuda.synchronize()
    g_used = OB.sigmoid(dt) if use_sig else d["g"]
    o_rec, s_ref = OD.forward(d["v"], d["b"], d["c"], g_used, d["A_log"], d["initial_state"])
    o_ref = OB.epilogue(o_rec, d["v"], D_skip if use_skip else np.zeros(H),
                        gate if use_gate else np.ones((B, T, H)))
    to, ts = TOL[DT[dtype]]
    assert rel(o.double().cpu().numpy(), o_ref) <= to
    assert rel(s.double().cpu().numpy(), s_ref) <= ts


def test_block_chain_conv_then_recurrence():
    """Prologue and recurrence chained as in the block (section 5.5, steps 2,
    5, 6): v = silu(conv(v_in)) feeds the recurrence and the skip; b, c, the
    decay logits and the output gate are random stand-ins for the projections."""
    B, T, H, S, Dh, K = 2, 500, 4, 32, 32, 4
    rng = np.random.default_rng(77)
    v_in = torch.from_numpy(rng.standard_normal((B, T, H * Dh))).to(torch.bfloat16)
    wc = torch.from_numpy(rng.standard_normal((H * Dh, K)) * 0.5).to(torch.float32)
    b = torch.from_numpy(rng.standard_normal((B, T, H, S)) / np.sqrt(S)).to(torch.bfloat16)
    c = torch.from_numpy(rng.standard_normal((B, T, H, S)) / np.sqrt(S)).to(torch.bfloat16)
    dt = torch.from_numpy(rng.standard_normal((B, T, H))).to(torch.float32)
    A_log = torch.from_numpy(rng.uniform(-2, 1, (H, S))).to(torch.float32)
    D_skip = torch.ones(H, dtype=torch.float32)
    gate = torch.from_numpy(OB.sigmoid(rng.standard_normal((B, T, H)))).to(torch.float32)
    v = G.gdn_conv_silu(v_in.cuda(), wc.cuda())
    o, s = G.gdn_diag_fwd(v.view(B, T, H, Dh), b.cuda(), c.cuda(), dt.cuda(), A_log.cuda(),
                          D_skip=D_skip.cuda(), out_gate=gate.cuda(), gate_sigmoid=True,
                          check=True)
    torch.cuda.synchronize()
    # oracle chain, on the recurrence's own bf16 input v (the stored prologue output)
    v_ref, _ = OB.conv_silu(v_in, wc)
    assert rel(v.double().cpu().numpy(), v_ref) <= CONV_TOL["bf16"]
    v_stored = v.view(B, T, H, Dh).cpu()
    o_rec, s_ref = OD.forward(v_stored, b, c, OB.sigmoid(dt), A_log)
    o_ref = OB.epilogue(o_rec, v_stored, D_skip, gate)
    to, ts = TOL[torch.bfloat16]
    assert rel(o.double().cpu().numpy(), o_ref) <= to
    assert rel(s.double().cpu().numpy(), s_ref) <= ts
