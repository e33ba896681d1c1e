"""GPU test of gdn_fwd_static_scratch, the entry point for callers that
cannot allocate device memory (a plugin inside a framework that owns all
device allocations, a latency-critical loop where cudaMalloc could
synchronise the device, a process with a fixed memory budget).  It must give
the same results as gdn_fwd, call after call, while keeping its status record
in the library's own static device array instead of a caller workspace.

Collected last on purpose (file name), so a failing run that stops at the
first failure has already run every other test."""
import pytest
import torch

import parity
from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _dev(inp):
    return parity.to_dev(inp)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_static_scratch_matches_gdn_fwd_on_two_calls(dtype):
    if not torch.cuda.is_available():
        pytest.fail("CUDA not available")
    w = W.custom(B=2, T=300, H=4, dk=64, dv=128, dtype=dtype, init_state=True, seed=41)
    d = _dev(W.generate(w))
    o_ref, s_ref = G.gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                             check=True)
    tol_o, tol_s = parity.TOL[W._DTYPES[dtype]]
    # outputs are preallocated by the caller; the entry point allocates nothing
    o = torch.empty_like(o_ref)
    s = torch.empty_like(s_ref)
    # a warm-up call, so that the allocator and the library's set-up are settled
    assert G.gdn_fwd_static_scratch(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                    d["initial_state"], None, o, s, check=True) == 0
    torch.cuda.synchronize()
    for call in range(3):
        o.fill_(float("nan"))
        s.fill_(float("nan"))
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        free0 = torch.cuda.mem_get_info()[0]
        # the last call does not check: it only enqueues, then the caller syncs
        check = call < 2
        st = G.gdn_fwd_static_scratch(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                      d["initial_state"], None, o, s, check=check)
        assert st == 0, f"call {call}: {G.status_string(st)}"
        torch.cuda.synchronize()
        # no device memory was taken, by torch or by the library
        assert torch.cuda.memory_allocated() == alloc0, f"call {call}: torch allocated"
        assert torch.cuda.mem_get_info()[0] == free0, f"call {call}: device memory taken"
        assert parity.rel(o.double().cpu(), o_ref.double().cpu()) <= tol_o, f"call {call}: o"
        assert parity.rel(s.double().cpu(), s_ref.double().cpu()) <= tol_s, f"call {call}: state"


def test_static_scratch_reports_and_clears_device_errors():
    w = W.custom(B=1, T=40, H=2, dk=32, dv=32, dtype="fp32", seed=42)
    d = _dev(W.generate(w))
    o = torch.empty_like(d["v"])
    s = torch.empty((3, 2, 32, 32), dtype=torch.float32, device="cuda")
    bad = torch.tensor([0, 10, 9, 40], dtype=torch.int32, device="cuda")    # offsets decrease
    good = torch.tensor([0, 10, 25, 40], dtype=torch.int32, device="cuda")
    assert G.gdn_fwd_static_scratch(d["q"], d["k"], d["v"], d["g"], d["beta"], None, bad,
                                    o, s, check=True) == 6
    # the array kept the error; the next call must start from a clean status
    assert G.gdn_fwd_static_scratch(d["q"], d["k"], d["v"], d["g"], d["beta"], None, good,
                                    o, s, check=True) == 0
