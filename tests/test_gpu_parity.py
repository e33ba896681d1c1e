"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Relative L2 over whole tensors; bounds in parity.TOL."""
import numpy as np
import pytest
import torch

import oracle
import parity
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.fail("CUDA not available: the GPU tests need a GB300")
    G.lib()
    oracle.build()


def _check(inp, dtype, **kw):
    """Whole-tensor relative L2 within the bound of the storage dtype, and the
    worst single (sequence, head) unit within the same bound (a guard: one
    wrong unit among many barely moves the whole-tensor norm)."""
    ro, rs, o, s, uo, us = parity.compare(inp, gpu_kw=kw.get("gpu"), oracle_kw=kw.get("orc"),
                                          units=True)
    to, ts = parity.TOL[dtype]
    msg = (f"rel L2 o={ro:.3e} (<= {to}), state={rs:.3e} (<= {ts}); worst unit "
           f"o={uo:.3e}, state={us:.3e}")
    assert ro <= to and rs <= ts, msg
    assert uo <= to and us <= ts, msg
    return ro, rs, uo, us


# ---------------- the five named workloads, full size ----------------
@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_workload_full_size(name):
    w = W.WORKLOADS[name]
    inp = W.generate(w)
    ro, rs, uo, us = _check(inp, W._DTYPES[w.dtype])
    kernel = G.gdn_fwd_kernel_name(w.dk, w.dv, W._DTYPES[w.dtype])
    parity.MARGINS.append(f"{name} [{kernel}]: rel L2 o={ro:.3e} state={rs:.3e}; worst "
                          f"(sequence, head) o={uo:.3e} state={us:.3e}; bounds "
                          f"{parity.TOL[W._DTYPES[w.dtype]]}")


@pytest.mark.parametrize("name", ["hymo_bf16", "wide_bf16"])
def test_workload_full_size_simt(name):
    """The fp32 CUDA-core kernel on the bf16 workloads (forced)."""
    w = W.WORKLOADS[name]
    inp = W.generate(w)
    _check(inp, torch.bfloat16, gpu=dict(force_simt=True))


# ---------------- edge cases: ragged tails, tiny T, head-dim mixes ----------------
SHAPES = [(1, 1, 1, 32, 32), (1, 63, 2, 64, 64), (2, 64, 1, 32, 64), (1, 65, 2, 64, 32),
          (2, 130, 3, 128, 64), (1, 200, 2, 32, 256), (1, 129, 1, 128, 256),
          (3, 77, 2, 64, 128), (1, 1000, 1, 128, 128)]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,H,dk,dv", SHAPES)
@pytest.mark.parametrize("init", [False, True])
def test_edge_shapes(dtype, B, T, H, dk, dv, init):
    w = W.custom(B=B, T=T, H=H, dk=dk, dv=dv, dtype=dtype, gate_scale=1.0,
                 init_state=init, seed=1000 + T + dk + dv)
    _check(W.generate(w), W._DTYPES[dtype])


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_varlen_small(dtype):
    lens = [1, 63, 64, 65, 2, 300, 17]
    w = W.custom(num_seqs=len(lens), len_range=(1, 300), H=3, dk=64, dv=96, dtype=dtype,
                 init_state=True, seed=21)
    _check(W.generate(w, lengths=lens), W._DTYPES[dtype])


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_varlen_bitwise_equals_separate_runs(dtype):
    lens = [5, 64, 129, 1, 250]
    w = W.custom(num_seqs=len(lens), len_range=(1, 300), H=2, dk=128, dv=64, dtype=dtype,
                 init_state=True, seed=22)
    inp = W.generate(w, lengths=lens)
    o, s = parity.gpu_forward(inp)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        part = {"q": inp["q"][:, a:b].contiguous(), "k": inp["k"][:, a:b].contiguous(),
                "v": inp["v"][:, a:b].contiguous(), "g": inp["g"][:, a:b].contiguous(),
                "beta": inp["beta"][:, a:b].contiguous(),
                "initial_state": inp["initial_state"][n:n + 1].contiguous(),
                "cu_seqlens": None}
        o1, s1 = parity.gpu_forward(part)
        assert torch.equal(o1, o[:, a:b]), f"sequence {n}: o differs"
        assert torch.equal(s1, s[n:n + 1]), f"sequence {n}: final state differs"


def test_qk_l2norm_flag():
    w = W.custom(B=2, T=150, H=2, dk=64, dv=64, dtype="fp32", seed=23)
    inp = W.generate(w)
    scale = torch.rand(2, 150, 2, 1) * 5 + 0.5
    inp["q"] = (inp["q"] * scale).contiguous()
    inp["k"] = (inp["k"] * scale.flip(1)).contiguous()
    _check(inp, torch.float32, gpu=dict(qk_l2norm=True), orc=dict(qk_l2norm=True))


def test_beta_zero_closed_form_on_gpu():
    # gentle gates keep exp(sum g) inside fp32 range over the 300 tokens
    w = W.custom(B=1, T=300, H=2, dk=64, dv=64, dtype="fp32", init_state=True,
                 gate_scale=0.02, seed=24)
    inp = W.generate(w)
    inp["beta"] = torch.zeros_like(inp["beta"])
    o, s = parity.gpu_forward(inp)
    G_ = torch.cumsum(inp["g"].double(), dim=1)
    H0 = inp["initial_state"].double()
    o_ref = torch.exp(G_)[..., None] * torch.einsum("bhkd,bthk->bthd", H0, inp["q"].double())
    s_ref = torch.exp(G_[:, -1])[..., None, None] * H0
    assert parity.rel(o.double().cpu(), o_ref) < 1e-4
    assert parity.rel(s.double().cpu(), s_ref) < 1e-4


def test_golden_two_token_on_gpu():
    """The hand-worked example of tests/golden, embedded in dk = dv = 32 with zeros."""
    import json, os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                       "two_token_hand.json")))
    q = torch.zeros(1, 2, 1, 32); k = torch.zeros(1, 2, 1, 32); v = torch.zeros(1, 2, 1, 32)
    q[0, :, 0, :2] = torch.tensor(gold["q"]); k[0, :, 0, :2] = torch.tensor(gold["k"])
    v[0, :, 0, :2] = torch.tensor(gold["v"])
    g = torch.log(torch.tensor(gold["alpha"], dtype=torch.float32)).view(1, 2, 1)
    beta = torch.tensor(gold["beta"], dtype=torch.float32).view(1, 2, 1)
    inp = {"q": q, "k": k, "v": v, "g": g, "beta": beta, "initial_state": None,
           "cu_seqlens": None}
    o, s = parity.gpu_forward(inp)
    assert np.allclose(o[0, :, 0, :2].cpu().numpy(), gold["o"], rtol=1e-5, atol=1e-6)
    assert np.allclose(s[0, 0, :2, :2].cpu().numpy(), gold["final_state_dk_by_dv"],
                       rtol=1e-5, atol=1e-6)
    assert float(o[..., 2:].abs().max()) == 0.0


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_state_chaining_and_in_place(dtype):
    w = W.custom(B=2, T=300, H=2, dk=64, dv=64, dtype=dtype, init_state=True, seed=25)
    inp = parity.to_dev(W.generate(w))
    o, s = G.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                     inp["initial_state"], check=True)
    T1 = 100
    state = inp["initial_state"].clone()
    parts = []
    for a, b in ((0, T1), (T1, 300)):
        sl = lambda x: x[:, a:b].contiguous()
        oo, _ = G.gdn_fwd(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]),
                          sl(inp["beta"]), state, final_state=state, check=True)  # in place
        parts.append(oo)
    to, ts = parity.TOL[W._DTYPES[dtype]]
    assert parity.rel(torch.cat(parts, 1).double().cpu(), o.double().cpu()) < to
    assert parity.rel(state.double().cpu(), s.double().cpu()) < ts


def test_no_final_state():
    w = W.custom(B=1, T=70, H=1, dk=32, dv=32, dtype="bf16", seed=26)
    inp = parity.to_dev(W.generate(w))
    o1, s1 = G.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], check=True)
    o2, s2 = G.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                       output_final_state=False, check=True)
    assert s2 is None and torch.equal(o1, o2)


@pytest.mark.parametrize("cu", [[0, 10, 9, 40], [0, 30, 20, 40], [0, 10, 20, 39], [1, 10, 20, 40]])
def test_bad_seqlens_reported(cu):
    """Malformed offsets are found on the device and reported by gdn_check;
    the affected sequences write nothing."""
    w = W.custom(B=1, T=40, H=2, dk=32, dv=32, dtype="fp32", seed=27)
    inp = parity.to_dev(W.generate(w))
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    ws = G.new_workspace(3, 2, 32, 32)
    o = torch.full_like(inp["v"], 7.0)
    G.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, cu_t, o=o,
              workspace=ws)
    assert G.gdn_check(ws) == 6
    assert G.gdn_check(ws) == 0  # the check cleared the status word


# ---------------- chunk-size variants (32 and 128: the tensor-core variants for bf16
# with head_dim_k 64 and dv a multiple of 64, the fp32 CUDA-core kernel otherwise) ----------------
CHUNK_SHAPES = [(1, 1, 1, 32, 32), (2, 31, 2, 64, 64), (1, 32, 1, 32, 64), (1, 33, 2, 64, 32),
                (2, 127, 2, 32, 96), (1, 128, 1, 64, 64), (1, 129, 2, 64, 128),
                (2, 300, 3, 128, 64), (1, 1000, 1, 64, 64)]


@pytest.mark.parametrize("chunk", [32, 128])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,H,dk,dv", CHUNK_SHAPES)
def test_chunk_size_variants(chunk, dtype, B, T, H, dk, dv):
    if chunk == 128 and dk == 128:
        pytest.skip("128-token chunks with dk = 128 are not supported")
    w = W.custom(B=B, T=T, H=H, dk=dk, dv=dv, dtype=dtype, gate_scale=1.0, init_state=True,
                 seed=2000 + T + dk + dv + chunk)
    _check(W.generate(w), W._DTYPES[dtype], gpu=dict(chunk_size=chunk))


@pytest.mark.parametrize("chunk", [32, 128])
def test_chunk_size_variants_varlen(chunk):
    lens = [1, 31, 32, 33, 127, 128, 129, 300]
    w = W.custom(num_seqs=len(lens), len_range=(1, 300), H=2, dk=64, dv=64, dtype="bf16",
                 init_state=True, seed=31 + chunk)
    _check(W.generate(w, lengths=lens), torch.bfloat16, gpu=dict(chunk_size=chunk))


@pytest.mark.parametrize("chunk", [32, 128])
def test_chunk_size_variants_full_size(chunk):
    """The HyMo-shaped bench workload (B=8, T=4096, H=16, dk=dv=64) in 32- and
    128-token chunks."""
    w = W.WORKLOADS["hymo_bf16"]
    _check(W.generate(w), torch.bfloat16, gpu=dict(chunk_size=chunk))


def test_chunk_sizes_agree():
    """The result does not depend on the chunk size beyond rounding."""
    w = W.custom(B=2, T=500, H=2, dk=64, dv=64, dtype="fp32", gate_scale=1.0, init_state=True,
                 seed=41)
    inp = W.generate(w)
    outs = [parity.gpu_forward(inp, chunk_size=c) for c in (32, 64, 128)]
    for o, s in outs[1:]:
        assert parity.rel(o.double().cpu().numpy(), outs[0][0].double().cpu().numpy()) <= 1e-5
        assert parity.rel(s.double().cpu().numpy(), outs[0][1].double().cpu().numpy()) <= 1e-5


# ---------------- empty inputs ----------------
@pytest.mark.parametrize("dtype,dk,dv", [("fp32", 64, 64), ("bf16", 64, 64), ("bf16", 128, 128)])
def test_varlen_empty_sequences(dtype, dk, dv):
    """Empty sequences (equal offsets) are legal: they read nothing and their
    final state is their initial state, bit for bit."""
    lens = [5, 0, 70, 0, 64, 0]
    w = W.custom(num_seqs=len(lens), len_range=(0, 70), H=2, dk=dk, dv=dv, dtype=dtype,
                 init_state=True, seed=28)
    inp = W.generate(w, lengths=lens)
    ro, rs, _, s = parity.compare(inp)
    to, ts = parity.TOL[W._DTYPES[dtype]]
    assert ro <= to and rs <= ts, (ro, rs)
    for n in (1, 3, 5):
        assert torch.equal(s[n].cpu(), inp["initial_state"][n])


@pytest.mark.parametrize("varlen", [False, True])
@pytest.mark.parametrize("init", [False, True])
def test_zero_tokens(varlen, init):
    """A call with no tokens reads nothing and passes every state through
    (zeros without an initial state)."""
    N, H, dk, dv = 3, 2, 64, 64
    B = 1 if varlen else N
    bf = dict(dtype=torch.bfloat16, device="cuda")
    q = torch.empty((B, 0, H, dk), **bf)
    v = torch.empty((B, 0, H, dv), **bf)
    g = torch.empty((B, 0, H), dtype=torch.float32, device="cuda")
    beta = torch.empty((B, 0, H), **bf)
    cu = torch.zeros(N + 1, dtype=torch.int32, device="cuda") if varlen else None
    s0 = torch.randn((N, H, dk, dv), device="cuda") if init else None
    o, s = G.gdn_fwd(q, q, v, g, beta, s0, cu, check=True)
    assert o.numel() == 0
    assert torch.equal(s, s0 if init else torch.zeros_like(s))


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 64, 64), ("bf16", 128, 128), ("fp32", 64, 64)])
def test_varlen_many_short_sequences(dtype, dk, dv):
    """5000 packed sequences of 0 to 5 tokens (empty ones included): a large
    grid of mostly single-chunk sequences."""
    rng = np.random.default_rng(29)
    lens = rng.integers(0, 6, 5000).tolist()
    w = W.custom(num_seqs=len(lens), len_range=(0, 5), H=2, dk=dk, dv=dv, dtype=dtype,
                 init_state=True, seed=30)
    inp = W.generate(w, lengths=lens)
    ro, rs, _, _ = parity.compare(inp)
    to, ts = parity.TOL[W._DTYPES[dtype]]
    assert ro <= to and rs <= ts, (ro, rs)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128)])
def test_long_sequence_with_one_token_tail(dk, dv):
    """T = 64k + 1: 1024 full chunks and a one-token last chunk."""
    w = W.custom(B=1, T=65537, H=1, dk=dk, dv=dv, dtype="bf16", gate_scale=0.01,
                 init_state=True, seed=32)
    _check(W.generate(w), torch.bfloat16)


def _guarded(shape, dtype, guard=4096):
    """A tensor of `shape` inside a buffer with `guard` canary elements on each
    side (the view stays 16-byte aligned)."""
    n = int(np.prod(shape))
    buf = torch.full((guard + n + guard,), -1234.5, dtype=dtype, device="cuda")
    return buf, buf[guard:guard + n].view(shape)


def _guards_intact(buf, guard=4096):
    return bool(torch.all(buf[:guard] == -1234.5)) and bool(torch.all(buf[-guard:] == -1234.5))


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 64, 64), ("bf16", 128, 128), ("fp32", 64, 96)])
def test_outputs_stay_inside_their_buffers(dtype, dk, dv):
    """Canary regions around o and the final state are untouched: no kernel
    writes outside its outputs (ragged varlen tails included)."""
    lens = [1, 63, 65, 0, 130, 7]
    w = W.custom(num_seqs=len(lens), len_range=(0, 130), H=2, dk=dk, dv=dv, dtype=dtype,
                 init_state=True, seed=33)
    inp = parity.to_dev(W.generate(w, lengths=lens))
    tdt = W._DTYPES[dtype]
    obuf, o = _guarded(inp["v"].shape, tdt)
    sbuf, s = _guarded(inp["initial_state"].shape, torch.float32)
    G.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"],
              inp["cu_seqlens"], o=o, final_state=s, check=True)
    torch.cuda.synchronize()
    assert _guards_intact(obuf) and _guards_intact(sbuf)
    o_ref, s_ref = parity.oracle_forward(W.generate(w, lengths=lens))
    to, ts = parity.TOL[tdt]
    assert parity.rel(o.double().cpu().numpy(), o_ref) <= to
    assert parity.rel(s.double().cpu().numpy(), s_ref) <= ts


# ---------------- GDN_SEQ_SPLIT: long dense sequences cut into segments ----------------
@pytest.mark.parametrize("B,T,H,dv,init,l2,gs", [(1, 2000, 2, 128, True, False, 1e-3),
                                                  (1, 2000, 2, 128, False, True, 0.0),
                                                  (1, 4097, 1, 256, True, False, 1e-3),
                                                  (1, 777, 3, 128, True, False, 1e-3),
                                                  (2, 1500, 1, 128, True, False, 1e-3),
                                                  (1, 1700, 1, 192, True, False, 1e-3),
                                                  (1, 600, 2, 128, True, False, 1e-3),
                                                  (2, 1700, 1, 128, True, False, 1e-3),
                                                  (2, 4096, 8, 128, True, False, 1e-3)])
def test_seq_split(B, T, H, dv, init, l2, gs):
    """A split call equals the oracle within the bf16 bounds and the unsplit
    call up to rounding; with dk = 128 and few units the call takes 2 to 8
    segments.  On 152 SMs the last two cases give the first segment more
    chunks than the later ones (7 against 5 with a ragged last chunk; 24
    against 8 with 8 heads), each with two sequences.
    The gates are slow (gs = 0 is the plain delta rule) so that a segment's
    map M keeps weight: with fast gates M underflows to zero and the split
    result is the unsplit one bit for bit."""
    w = W.custom(B=B, T=T, H=H, dk=128, dv=dv, dtype="bf16", init_state=init, gate_scale=gs,
                 seed=700 + T + dv)
    assert G.gdn_fwd_split_segments(B, T, H, 128, dv, torch.bfloat16, G.GDN_SEQ_SPLIT) > 1
    inp = W.generate(w)
    kw = dict(qk_l2norm=True) if l2 else {}
    if l2:
        ex = W.generate_block_extras(inp, H, seed=701)
        inp = dict(inp, q=ex["q_raw"], k=ex["k_raw"])
    d = parity.to_dev(inp)
    o0, s0 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                       check=True, **kw)
    o1, s1 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                       check=True, seq_split=True, **kw)
    o_ref, s_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["initial_state"], None, qk_l2norm=l2)
    o64, s64 = o1.double().cpu().numpy(), s1.double().cpu().numpy()
    to, ts = parity.TOL[torch.bfloat16]
    assert parity.rel(o64, o_ref) <= to and parity.rel(s64, s_ref) <= ts
    assert parity.worst_unit_state(s64, s_ref) <= ts
    # close to the unsplit call (the segments' maps add bf16 operand rounding)
    assert parity.rel(o64, o0.double().cpu().numpy()) <= 5e-3
    assert parity.rel(s64, s0.double().cpu().numpy()) <= 5e-3
    assert not torch.equal(s0, s1)  # the split path ran (its composition rounds differently)


def test_seq_split_with_epilogue_runs_unsplit():
    """The block epilogue is not combined with a split: such a call runs
    unsplit (same result as without the flag, bit for bit)."""
    w = W.custom(B=1, T=2000, H=2, dk=128, dv=128, dtype="bf16", init_state=True,
                 gate_scale=1e-3, seed=31)
    inp = W.generate(w)
    ex = W.generate_block_extras(inp, w.H, seed=32)
    d = parity.to_dev(inp)
    kw = dict(D_skip=ex["D_skip"].cuda(), out_gate=ex["out_gate"].cuda(), check=True)
    o0, s0 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None, **kw)
    o1, s1 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                       seq_split=True, **kw)
    assert torch.equal(o0, o1) and torch.equal(s0, s1)


def test_seq_split_long_full_size():
    """long_bf16 (B=1, T=65536, H=16, dk=dv=128, slow gates) split into segments,
    against the oracle on the whole tensors and the worst (sequence, head)."""
    w = W.WORKLOADS["long_bf16"]
    inp = W.generate(w)
    d = parity.to_dev(inp)
    o, s = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                     check=True, seq_split=True)
    o_ref, s_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["initial_state"], None)
    o64, s64 = o.double().cpu().numpy(), s.double().cpu().numpy()
    ro, rs = parity.rel(o64, o_ref), parity.rel(s64, s_ref)
    uo, us = parity.worst_unit_o(o64, o_ref, None), parity.worst_unit_state(s64, s_ref)
    parity.MARGINS.append(f"long_bf16 split into segments [tc128_bf16]: rel L2 o={ro:.3e} "
                          f"state={rs:.3e}; worst (sequence, head) o={uo:.3e} state={us:.3e}")
    to, ts = parity.TOL[torch.bfloat16]
    assert ro <= to and rs <= ts and uo <= to and us <= ts


def _split_makespan(a, b, first, seg, sms):
    """Chunk steps of one launch that dispatches a CTAs of `first` chunks and
    then b of `seg` chunks on sms SMs, each CTA to the first SM that frees
    (the sms - a SMs left free start at 0, the other a at `first`)."""
    free, done, rf, ra, last = sms - a, 0, 0, 0, 0
    while done < b:
        tf = rf * seg if free > 0 else float("inf")
        ta = first + ra * seg
        if tf <= ta:
            done, last, rf = done + free, tf, rf + 1
        else:
            done, last, ra = done + a, ta, ra + 1
    return max(first, last + seg)


def _expected_segments(N, T, H, dv, sms):
    """The documented plan rule: the later segments are of equal length
    chunks / (k + S - 1) (at least 4 chunks), the first takes the rest; over S
    = 2 .. 8 and k = 1 .. 16 take the shortest launch (the first segments'
    value tiles dispatched first, then each later segment's value and
    transport tiles, one CTA per SM), the fewest segments among equals, and
    split only when that beats the unsplit launch by a quarter.  Calls whose
    first segments alone fill the SMs are not split."""
    a, u, chunks = N * H * dv // 64, N * H * (dv + 128) // 64, (T + 63) // 64
    if a >= sms:
        return 1
    best, best_span = 1, 0.75 * chunks
    for S in range(2, 9):
        for k in range(1, 17):
            seg = chunks // (k + S - 1)
            if seg < 4:
                break
            span = _split_makespan(a, (S - 1) * u, chunks - (S - 1) * seg, seg, sms)
            if span < best_span:
                best, best_span = S, span
    return best


def test_seq_split_plan():
    """The library's split plan on this device follows the documented rule:
    the long workload (16 units of two column tiles) is split, the wide one
    (128 units) fills the SMs unsplit, packed varlen calls and sequences of
    fewer than 8 chunks are never split."""
    S = G.gdn_fwd_split_segments
    bf = torch.bfloat16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for (N, T, H, dv) in [(1, 65536, 16, 128), (4, 8192, 16, 128), (1, 12 * 64, 1, 128),
                          (1, 4097, 1, 256), (2, 2000, 3, 128), (1, 600, 2, 128)]:
        assert S(N, T, H, 128, dv, bf, G.GDN_SEQ_SPLIT) == _expected_segments(N, T, H, dv, sms)
    assert S(1, 65536, 16, 128, 128, bf, G.GDN_SEQ_SPLIT) >= 2
    assert S(4, 8192, 16, 128, 128, bf, G.GDN_SEQ_SPLIT) == 1
    assert S(1, 140000, 8, 128, 256, bf, G.GDN_SEQ_SPLIT, varlen=True) == 1
    assert S(1, 7 * 64, 1, 128, 128, bf, G.GDN_SEQ_SPLIT) == 1   # under 8 chunks


def test_seq_split_needs_its_workspace():
    """A call the plan splits needs gdn_fwd_split_workspace_size bytes: one
    sized without the flag, or with it but without the token count, is
    refused before any launch."""
    w = W.custom(B=1, T=1000, H=2, dk=128, dv=128, dtype="bf16", init_state=True, seed=9)
    d = parity.to_dev(W.generate(w))
    assert G.gdn_fwd_split_segments(1, 1000, 2, 128, 128, torch.bfloat16, G.GDN_SEQ_SPLIT) > 1
    for small in (G.new_workspace(1, 2, 128, 128),
                  G.new_workspace(1, 2, 128, 128, G.GDN_SEQ_SPLIT)):
        with pytest.raises(G.GdnError):
            G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                      workspace=small, seq_split=True)
    ok = G.new_workspace(1, 2, 128, 128, G.GDN_SEQ_SPLIT, seq_len=1000)
    G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
              workspace=ok, seq_split=True, check=True)
