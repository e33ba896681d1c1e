"""GPU parity of the backward pass (``gdn_bwd``) against the fp64 autograd
oracle ``oracle.grad`` on the same seeded inputs, through the C ABI.

Two paths, two bounds (relative L2 over each whole gradient tensor):
- fp32 storage, and bf16 storage with head_dim_v = 256, run the token-serial
  fp32 backward; every gradient is computed in fp32 from the stored inputs,
  so it is held to 1e-4.
- bf16 storage with head_dim_k, head_dim_v <= 128 runs the chunked backward,
  whose products take bf16 operands with fp32 accumulation, as the forward's
  tensor-core path does; it is held to the forward's bf16 bound on o, 1e-2.
  (Rounding every product operand of the chunked algebra to bf16 in an fp64
  emulation gives 2e-3 to 4e-3 on these inputs.)"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.grad as OG
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W
from parity import rel

pytestmark = pytest.mark.gpu

GRAD_TOL = 1e-4
BF16_GRAD_TOL = 1e-2


def _tol(dtype, dk, dv):
    return BF16_GRAD_TOL if dtype == "bf16" and dk <= 128 and dv <= 128 else GRAD_TOL
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _dev(x):
    return None if x is None else x.cuda()


def _run(inp, d_o, dhN):
    gr = G.gdn_bwd(_dev(inp["q"]), _dev(inp["k"]), _dev(inp["v"]), _dev(inp["g"]),
                   _dev(inp["beta"]), _dev(d_o), _dev(inp["initial_state"]),
                   _dev(inp["cu_seqlens"]), _dev(dhN), check=True)
    torch.cuda.synchronize()
    return {k: v.double().cpu().numpy() for k, v in gr.items()}


def _ref(inp, d_o, dhN):
    return OG.backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                       inp["initial_state"], d_o, dhN, inp["cu_seqlens"])


def _upstream(inp, seed, with_dhN):
    rng = np.random.default_rng(seed)
    v = inp["v"]
    d_o = torch.from_numpy(rng.standard_normal(tuple(v.shape))).to(v.dtype)
    dhN = None
    if with_dhN:
        N, H = inp["N"], v.shape[2]
        dhN = torch.from_numpy(rng.standard_normal((N, H, inp["q"].shape[-1], v.shape[-1]))
                               ).to(torch.float32)
    return d_o, dhN


def _check(gpu, ref, tol=GRAD_TOL):
    errs = {n: rel(gpu[n], ref[n]) for n in NAMES}
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"rel L2 above {tol}: {bad} (all: {errs})"


SHAPES = [(1, 1, 1, 32, 32), (1, 7, 2, 32, 32), (2, 64, 1, 64, 64), (1, 65, 2, 64, 32),
          (1, 130, 2, 32, 64), (2, 100, 2, 128, 64), (1, 200, 1, 64, 256),
          (1, 200, 2, 128, 128), (2, 70, 1, 128, 32), (1, 130, 2, 64, 128), (1, 100, 1, 32, 128)]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,H,dk,dv", SHAPES, ids=[f"B{b}T{t}H{h}k{k}v{v}" for b, t, h, k, v in SHAPES])
@pytest.mark.parametrize("init", [False, True])
def test_bwd_matches_oracle(dtype, B, T, H, dk, dv, init):
    w = W.custom(B=B, T=T, H=H, dk=dk, dv=dv, dtype=dtype, gate_scale=1.0, init_state=init,
                 seed=3000 + T + dk + dv)
    inp = W.generate(w)
    d_o, dhN = _upstream(inp, 7 + T, init)
    _check(_run(inp, d_o, dhN), _ref(inp, d_o, dhN), _tol(dtype, dk, dv))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_bwd_varlen(dtype):
    lens = [1, 63, 64, 65, 9, 140]
    w = W.custom(num_seqs=len(lens), len_range=(1, 140), H=2, dk=64, dv=64, dtype=dtype,
                 init_state=True, seed=51)
    inp = W.generate(w, lengths=lens)
    d_o, dhN = _upstream(inp, 52, True)
    _check(_run(inp, d_o, dhN), _ref(inp, d_o, dhN), _tol(dtype, 64, 64))


def test_bwd_slow_gates_long():
    """Slow decays (gate scale 0.01) over 1000 tokens: the gradient reaches far back."""
    w = W.custom(B=1, T=1000, H=2, dk=64, dv=64, dtype="bf16", gate_scale=0.01,
                 init_state=True, seed=53)
    inp = W.generate(w)
    d_o, dhN = _upstream(inp, 54, True)
    _check(_run(inp, d_o, dhN), _ref(inp, d_o, dhN), _tol("bf16", 64, 64))


def test_bwd_full_size_sampled():
    """The HyMo-shaped bench workload (B=8, T=4096, H=16, dk=dv=64, bf16) in one
    call; the oracle runs on sampled (batch row, head) pairs."""
    w = W.WORKLOADS["hymo_bf16"]
    inp = W.generate(w)
    d_o, _ = _upstream(inp, 55, False)
    gpu = _run(inp, d_o, None)
    for b, h in ((0, 0), (3, 7), (7, 15)):
        one = {n: inp[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        one.update(initial_state=None, cu_seqlens=None)
        ref = _ref(one, d_o[b:b + 1, :, h:h + 1], None)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            assert rel(gpu[n][b:b + 1, :, h:h + 1], ref[n]) <= BF16_GRAD_TOL, (n, b, h)
        assert rel(gpu["dh0"][b:b + 1, h:h + 1], ref["dh0"]) <= BF16_GRAD_TOL, ("dh0", b, h)


def test_bwd_chunk_checkpoints_only():
    """Many heads on the token-serial path (B=1, T=130, H=2048, dk=128, dv=256,
    bf16): the 8-token checkpoints would take more than 4 GiB, so the workspace
    holds one state per 64-token chunk and the backward recomputes the
    sub-chunk starts.  The oracle runs on sampled heads."""
    B, T, H, dk, dv = 1, 130, 2048, 128, 256
    fine = 3 * 8 * H * dk * dv * 4     # 3 chunks x 8 sub-chunk states
    assert G.gdn_bwd_workspace_size(B, T, H, dk, dv) < fine
    w = W.custom(B=B, T=T, H=H, dk=dk, dv=dv, dtype="bf16", gate_scale=1.0, init_state=True,
                 seed=57)
    inp = W.generate(w)
    d_o, dhN = _upstream(inp, 58, True)
    gr = G.gdn_bwd(_dev(inp["q"]), _dev(inp["k"]), _dev(inp["v"]), _dev(inp["g"]),
                   _dev(inp["beta"]), _dev(d_o), _dev(inp["initial_state"]), None, _dev(dhN),
                   check=True)
    torch.cuda.synchronize()
    for h in (0, 1234, 2047):
        one = {n: inp[n][:, :, h:h + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        one.update(initial_state=inp["initial_state"][:, h:h + 1].contiguous(), cu_seqlens=None)
        ref = _ref(one, d_o[:, :, h:h + 1].contiguous(), dhN[:, h:h + 1].contiguous())
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            got = gr[n][:, :, h:h + 1].double().cpu().numpy()
            assert rel(got, ref[n]) <= GRAD_TOL, (n, h)
        got = gr["dh0"][:, h:h + 1].double().cpu().numpy()
        assert rel(got, ref["dh0"]) <= GRAD_TOL, ("dh0", h)


def test_bwd_wide_sampled():
    """The wide workload (B=4, T=8192, H=16, dk=dv=128, bf16) on the chunked path
    in one call; the oracle runs on one sampled (batch row, head) pair."""
    w = W.WORKLOADS["wide_bf16"]
    inp = W.generate(w)
    d_o, _ = _upstream(inp, 59, False)
    gpu = _run(inp, d_o, None)
    b, h = 2, 11
    one = {n: inp[n][b:b + 1, :, h:h + 1].contiguous() for n in ("q", "k", "v", "g", "beta")}
    one.update(initial_state=inp["initial_state"][b:b + 1, h:h + 1].contiguous(), cu_seqlens=None)
    ref = _ref(one, d_o[b:b + 1, :, h:h + 1], None)
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        assert rel(gpu[n][b:b + 1, :, h:h + 1], ref[n]) <= BF16_GRAD_TOL, (n, b, h)
    assert rel(gpu["dh0"][b:b + 1, h:h + 1], ref["dh0"]) <= BF16_GRAD_TOL, ("dh0", b, h)


def test_bwd_varlen_dk128():
    """Packed sequences on the chunked path with head dims of 128."""
    lens = [1, 63, 64, 65, 9, 140]
    w = W.custom(num_seqs=len(lens), len_range=(1, 140), H=1, dk=128, dv=128, dtype="bf16",
                 init_state=True, seed=61)
    inp = W.generate(w, lengths=lens)
    d_o, dhN = _upstream(inp, 62, True)
    _check(_run(inp, d_o, dhN), _ref(inp, d_o, dhN), BF16_GRAD_TOL)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("cu", [[0, 10, 9, 40], [0, 30, 20, 40], [0, 10, 20, 39], [1, 10, 20, 40]])
def test_bwd_bad_seqlens_reported(dtype, cu):
    """Malformed offsets are found on the device by both backward paths and
    reported by gdn_check (GDN_ERR_BAD_SEQLENS), which then clears the word."""
    w = W.custom(B=1, T=40, H=2, dk=32, dv=32, dtype=dtype, seed=63)
    inp = W.generate(w)
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    q, k, v, g, beta = (inp[n].cuda() for n in ("q", "k", "v", "g", "beta"))
    d_o = torch.ones_like(v)
    ws = torch.zeros(G.gdn_bwd_workspace_size(3, 40, 2, 32, 32), dtype=torch.uint8, device="cuda")
    G.gdn_bwd(q, k, v, g, beta, d_o, None, cu_t, None, workspace=ws)
    assert G.gdn_check(ws) == 6
    assert G.gdn_check(ws) == 0


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_bwd_varlen_empty_sequences(dtype):
    """Empty sequences on both paths: no token gradients, and the gradient of
    their initial state is d_final_state."""
    lens = [5, 0, 70, 0, 64, 0]
    w = W.custom(num_seqs=len(lens), len_range=(0, 70), H=2, dk=64, dv=64, dtype=dtype,
                 init_state=True, seed=64)
    inp = W.generate(w, lengths=lens)
    d_o, dhN = _upstream(inp, 65, True)
    gpu = _run(inp, d_o, dhN)
    _check(gpu, _ref(inp, d_o, dhN), _tol(dtype, 64, 64))
    for n in (1, 3, 5):
        assert np.array_equal(gpu["dh0"][n], dhN[n].double().numpy())


def test_bwd_zero_tokens():
    """A call with no tokens passes d_final_state through to d initial_state."""
    N, H, dk, dv = 2, 2, 64, 64
    bf = dict(dtype=torch.bfloat16, device="cuda")
    q = torch.empty((N, 0, H, dk), **bf)
    v = torch.empty((N, 0, H, dv), **bf)
    g = torch.empty((N, 0, H), dtype=torch.float32, device="cuda")
    beta = torch.empty((N, 0, H), **bf)
    dhN = torch.randn((N, H, dk, dv), device="cuda")
    gr = G.gdn_bwd(q, q, v, g, beta, torch.empty_like(v), None, None, dhN, check=True)
    assert torch.equal(gr["dh0"], dhN)
    gr = G.gdn_bwd(q, q, v, g, beta, torch.empty_like(v), None, None, None, check=True)
    assert torch.equal(gr["dh0"], torch.zeros_like(dhN))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_bwd_varlen_many_short_sequences(dtype):
    """600 packed sequences of 0 to 5 tokens on both paths: every chunk slot of
    the chunked path is found by its binary search over the offsets."""
    rng = np.random.default_rng(66)
    lens = rng.integers(0, 6, 600).tolist()
    w = W.custom(num_seqs=len(lens), len_range=(0, 5), H=1, dk=64, dv=64, dtype=dtype,
                 init_state=True, seed=67)
    inp = W.generate(w, lengths=lens)
    d_o, dhN = _upstream(inp, 68, True)
    _check(_run(inp, d_o, dhN), _ref(inp, d_o, dhN), _tol(dtype, 64, 64))


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 64, 64), ("bf16", 128, 128), ("fp32", 64, 64)])
def test_bwd_outputs_stay_inside_their_buffers(dtype, dk, dv):
    """Canary regions around every gradient are untouched on both paths
    (ragged varlen tails and an empty sequence included)."""
    lens = [1, 63, 65, 0, 130]
    w = W.custom(num_seqs=len(lens), len_range=(0, 130), H=2, dk=dk, dv=dv, dtype=dtype,
                 init_state=True, seed=69)
    inp = W.generate(w, lengths=lens)
    d_o, dhN = _upstream(inp, 70, True)
    B, T, H = inp["q"].shape[:3]
    N = len(lens)
    guard = 4096
    shapes = {"dq": (B, T, H, dk), "dk": (B, T, H, dk), "dv": (B, T, H, dv), "dg": (B, T, H),
              "dbeta": (B, T, H), "dh0": (N, H, dk, dv)}
    bufs, grads = {}, {}
    for name, shp in shapes.items():
        n = int(np.prod(shp))
        bufs[name] = torch.full((guard + n + guard,), -1234.5, dtype=torch.float32, device="cuda")
        grads[name] = bufs[name][guard:guard + n].view(shp)
    G.gdn_bwd(_dev(inp["q"]), _dev(inp["k"]), _dev(inp["v"]), _dev(inp["g"]), _dev(inp["beta"]),
              _dev(d_o), _dev(inp["initial_state"]), _dev(inp["cu_seqlens"]), _dev(dhN),
              grads=grads, check=True)
    torch.cuda.synchronize()
    for name, buf in bufs.items():
        assert bool(torch.all(buf[:guard] == -1234.5)) and bool(torch.all(buf[-guard:] == -1234.5)), name
    ref = _ref(inp, d_o, dhN)
    _check({k: v.double().cpu().numpy() for k, v in grads.items()}, ref, _tol(dtype, dk, dv))
