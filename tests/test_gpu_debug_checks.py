"""GDN_DEBUG_CHECKS on the GPU: with the extents from the shapes every check
passes and the results are the plain kernels' bit for bit (and match the
oracle); with a declared extent smaller than what some blocks would touch,
exactly those blocks record GDN_ERR_DEVICE_CHECK with their (sequence, head)
and the buffer's site, and end without touching anything.  The declared
extents are deliberately undersized views of full-size buffers, so every real
access stays in bounds whatever the kernels do; no check can fault."""
import numpy as np
import pytest
import torch

import oracle
import parity
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SITE = {v: k for k, v in G.DEBUG_SITES.items()}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.fail("CUDA not available: the GPU tests need a GB300")
    G.lib()
    oracle.build()


# (B, T, H, dk, dv, dtype): the tc64, tc128 and fp32 CUDA-core kernels
CASES = [(4, 200, 2, 64, 64, "bf16"), (3, 130, 2, 128, 128, "bf16"), (3, 100, 2, 64, 64, "fp32")]


@pytest.mark.parametrize("chunk", [32, 128])
def test_debug_checks_on_the_chunk_variants(chunk):
    """The chunk-size variants run the same range checks: results unchanged
    with the checks on, and an undersized q extent caught for sequences 2.."""
    B, T, H, dk, dv = 4, 150, 2, 64, 64
    inp = make(B, T, H, dk, dv, "bf16")
    d = parity.to_dev(inp)
    o0, s0 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                       chunk_size=chunk, check=True)
    o1, s1 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                       chunk_size=chunk, check=True, debug_checks=True)
    assert torch.equal(o0, o1) and torch.equal(s0, s1)
    o, s = outputs_like(d, B, H, dk, dv)
    ws = G.new_workspace(B, H, dk, dv)
    assert G.gdn_fwd_debug(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                           o, s, ws, declared=dict(q=2 * T * H * dk),
                           chunk_size=chunk) == G.GDN_OK
    st, seq, head, site = G.gdn_check_record(ws)
    assert st == G.GDN_ERR_DEVICE_CHECK and seq >= 2 and site == SITE["q"]
    assert torch.equal(o[:2], o0[:2]) and torch.isnan(o[2:].float()).all()


def make(B, T, H, dk, dv, dtype, seed=11, varlen=None):
    if varlen is None:
        w = W.custom(name="dbg", B=B, T=T, H=H, dk=dk, dv=dv, dtype=dtype, init_state=True,
                     seed=seed)
        return W.generate(w)
    w = W.custom(name="dbg", num_seqs=len(varlen), len_range=(1, 8), H=H, dk=dk, dv=dv,
                 dtype=dtype, init_state=True, seed=seed)
    return W.generate(w, lengths=varlen)


def outputs_like(d, N, H, dk, dv):
    o = torch.full_like(d["v"], float("nan"))
    s = torch.full((N, H, dk, dv), float("nan"), dtype=torch.float32, device=d["v"].device)
    return o, s


@pytest.mark.parametrize("B,T,H,dk,dv,dtype", CASES)
def test_debug_checks_pass_and_change_nothing(B, T, H, dk, dv, dtype):
    inp = make(B, T, H, dk, dv, dtype)
    d = parity.to_dev(inp)
    o0, s0 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                       check=True)
    o1, s1 = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                       check=True, debug_checks=True)
    assert torch.equal(o0, o1) and torch.equal(s0, s1)
    # the shape-derived extents through the explicit entry point, too
    N = B
    o2, s2 = outputs_like(d, N, H, dk, dv)
    ws = G.new_workspace(N, H, dk, dv)
    assert G.gdn_fwd_debug(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                           o2, s2, ws) == G.GDN_OK
    assert G.gdn_check_record(ws) == (G.GDN_OK, -1, -1, 0)
    assert torch.equal(o0, o2) and torch.equal(s0, s2)
    o_ref, s_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["initial_state"], None)
    to, ts = parity.TOL[W._DTYPES[dtype]]
    assert parity.rel(o1.double().cpu().numpy(), o_ref) <= to
    assert parity.rel(s1.double().cpu().numpy(), s_ref) <= ts


@pytest.mark.parametrize("B,T,H,dk,dv,dtype", CASES)
@pytest.mark.parametrize("buf", ["q", "k", "v", "g", "beta", "o", "initial_state",
                                 "final_state"])
def test_undersized_extent_is_caught_before_use(B, T, H, dk, dv, dtype, buf):
    """Declare each buffer as holding only the first two sequences' rows (or
    states): the blocks of sequences 2.. record the buffer's site and write
    nothing; sequences 0 and 1 are computed as usual."""
    inp = make(B, T, H, dk, dv, dtype)
    d = parity.to_dev(inp)
    N = B
    ref_o, ref_s = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                             None, check=True)
    per_row = dict(q=dk, k=dk, v=dv, o=dv, g=1, beta=1)
    if buf in per_row:
        declared = {buf: 2 * T * H * per_row[buf]}
    else:
        declared = {buf: 2 * H * dk * dv}
    o, s = outputs_like(d, N, H, dk, dv)
    ws = G.new_workspace(N, H, dk, dv)
    assert G.gdn_fwd_debug(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                           o, s, ws, declared=declared) == G.GDN_OK
    st, seq, head, site = G.gdn_check_record(ws)
    assert st == G.GDN_ERR_DEVICE_CHECK, G.status_string(st)
    assert seq >= 2 and 0 <= head < H and site == SITE[buf], (seq, head, site)
    # sequences 0, 1: the plain result; 2..: untouched (still the NaN fill)
    assert torch.equal(o[:2], ref_o[:2]) and torch.equal(s[:2], ref_s[:2])
    assert torch.isnan(o[2:].float()).all() and torch.isnan(s[2:]).all()
    # the status was cleared by the read
    assert G.gdn_check(ws) == G.GDN_OK


def test_undersized_out_gate_extent():
    B, T, H, dk, dv = 3, 160, 2, 64, 64
    inp = make(B, T, H, dk, dv, "bf16")
    ex = W.generate_block_extras(inp, H, seed=4)
    d = parity.to_dev(inp)
    e = parity.to_dev(ex)
    o, s = outputs_like(d, B, H, dk, dv)
    ws = G.new_workspace(B, H, dk, dv)
    assert G.gdn_fwd_debug(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                           o, s, ws, D_skip=e["D_skip"], out_gate=e["out_gate"],
                           declared=dict(out_gate=T * H)) == G.GDN_OK
    st, seq, head, site = G.gdn_check_record(ws)
    assert (st, site) == (G.GDN_ERR_DEVICE_CHECK, SITE["out_gate"]) and seq >= 1
    ref_o, ref_s = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], None,
                             D_skip=e["D_skip"], out_gate=e["out_gate"], check=True)
    assert torch.equal(o[:1], ref_o[:1]) and torch.equal(s[:1], ref_s[:1])
    assert torch.isnan(o[1:].float()).all()


def test_undersized_extent_varlen():
    """Packed sequences: the v extent ends inside sequence 1, so sequence 1 and
    every later one record the v site; sequence 0 is computed."""
    H, dk, dv = 2, 64, 64
    inp = make(1, 0, H, dk, dv, "bf16", varlen=[150, 90, 0, 200])
    d = parity.to_dev(inp)
    cu = inp["cu_seqlens"].tolist()
    N = len(cu) - 1
    ref_o, ref_s = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                             d["cu_seqlens"], check=True)
    o, s = outputs_like(d, N, H, dk, dv)
    ws = G.new_workspace(N, H, dk, dv)
    cut = (cu[1] + 10) * H * dv
    assert G.gdn_fwd_debug(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                           d["cu_seqlens"], o, s, ws, declared=dict(v=cut)) == G.GDN_OK
    st, seq, head, site = G.gdn_check_record(ws)
    assert (st, site) == (G.GDN_ERR_DEVICE_CHECK, SITE["v"]) and seq in (1, 3), seq
    assert torch.equal(o[:, :cu[1]], ref_o[:, :cu[1]]) and torch.equal(s[0], ref_s[0])
    assert torch.isnan(o[:, cu[1]:].float()).all()
    # the empty sequence 2 touches no token buffer: its state passes through
    assert torch.equal(s[2], ref_s[2])
    assert torch.isnan(s[1]).all() and torch.isnan(s[3]).all()
