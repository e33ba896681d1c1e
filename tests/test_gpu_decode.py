"""GPU parity of the decode entry point (one recurrent step per sequence)
against the oracle's token-by-token recurrence, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W
from parity import TOL, rel

pytestmark = pytest.mark.gpu

# fp32 arithmetic on the state in both storage dtypes: the state is compared
# at this bound; o at the storage-dtype bound of the prefill tests.
STATE_TOL = 1e-5


def _dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _oracle_step(d, qk_l2norm=False):
    """The oracle on the same values as a batch of one-token sequences."""
    q, k, v = d["q"][:, None], d["k"][:, None], d["v"][:, None]
    g, beta = d["g"][:, None], d["beta"][:, None]
    return oracle.forward(q, k, v, g, beta, d["state"], None, qk_l2norm=qk_l2norm)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (64, 96), (128, 128), (128, 256)])
@pytest.mark.parametrize("init", [False, True])
def test_decode_step_matches_oracle(dtype, dk, dv, init):
    w = W.custom(B=5, T=1, H=3, dk=dk, dv=dv, dtype=dtype, init_state=init, seed=dk + dv)
    d = W.generate_decode(w)
    o, s = G.gdn_decode(**{k: v for k, v in _dev(d).items() if k != "N"})
    torch.cuda.synchronize()
    o_ref, s_ref = _oracle_step(d)
    tol_o = TOL[W._DTYPES[dtype]][0]
    assert rel(o.double().cpu().numpy()[:, None], o_ref) <= tol_o
    assert rel(s.double().cpu().numpy(), s_ref) <= STATE_TOL


def test_decode_l2norm_matches_oracle():
    w = W.custom(B=4, T=1, H=2, dk=64, dv=64, dtype="fp32", init_state=True, seed=11)
    d = W.generate_decode(w)
    d["q"] = d["q"] * 3.0 + 0.1
    d["k"] = d["k"] * 0.5
    o, s = G.gdn_decode(**{k: v for k, v in _dev(d).items() if k != "N"}, qk_l2norm=True)
    torch.cuda.synchronize()
    o_ref, s_ref = _oracle_step(d, qk_l2norm=True)
    assert rel(o.double().cpu().numpy()[:, None], o_ref) <= 1e-5
    assert rel(s.double().cpu().numpy(), s_ref) <= STATE_TOL


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_chain_equals_the_recurrence(dtype):
    """T steps, the state updated in place, against the oracle over the T tokens."""
    T = 24
    w = W.custom(B=3, T=T, H=2, dk=64, dv=64, dtype=dtype, init_state=True, seed=5)
    d = W.generate(w)
    dd = _dev(d)
    state = dd["initial_state"].clone()
    outs = []
    for t in range(T):
        o, st = G.gdn_decode(dd["q"][:, t].contiguous(), dd["k"][:, t].contiguous(),
                             dd["v"][:, t].contiguous(), dd["g"][:, t].contiguous(),
                             dd["beta"][:, t].contiguous(), state, state_out=state)
        assert st.data_ptr() == state.data_ptr()
        outs.append(o)
    torch.cuda.synchronize()
    o_gpu = torch.stack(outs, dim=1).double().cpu().numpy()
    o_ref, s_ref = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  d["initial_state"], None)
    assert rel(o_gpu, o_ref) <= TOL[W._DTYPES[dtype]][0]
    assert rel(state.double().cpu().numpy(), s_ref) <= 1e-4


def test_decode_agrees_with_the_prefill_path_on_one_token():
    w = W.custom(B=6, T=1, H=4, dk=64, dv=64, dtype="bf16", init_state=True, seed=3)
    d = W.generate(w)
    dd = _dev(d)
    o1, s1 = G.gdn_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["initial_state"],
                       None, check=True)
    o2, s2 = G.gdn_decode(dd["q"][:, 0].contiguous(), dd["k"][:, 0].contiguous(),
                          dd["v"][:, 0].contiguous(), dd["g"][:, 0].contiguous(),
                          dd["beta"][:, 0].contiguous(), dd["initial_state"])
    torch.cuda.synchronize()
    assert rel(o2.double().cpu().numpy(), o1[:, 0].double().cpu().numpy()) <= 1e-2
    assert rel(s2.double().cpu().numpy(), s1.double().cpu().numpy()) <= 5e-3


def test_decode_full_size_sampled():
    """The bench's decode workload: 1024 sequences x 16 heads, checked on a
    sample of (sequence, head) pairs against the oracle."""
    w = W.DECODE_WORKLOADS["decode_hymo_bf16"]
    d = W.generate_decode(w)
    o, s = G.gdn_decode(**{k: v for k, v in _dev(d).items() if k != "N"})
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(w.B, 16, replace=False)
    sub = {k: (v[rows] if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    o_ref, s_ref = _oracle_step(sub)
    assert rel(o[rows].double().cpu().numpy()[:, None], o_ref) <= 1e-2
    assert rel(s[rows].double().cpu().numpy(), s_ref) <= STATE_TOL
