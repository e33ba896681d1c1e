"""Failure reporting on the GPU without faulting it: a bounded device-side
wait that nothing completes gives up and reports GDN_ERR_TIMEOUT through the
workspace status word, and the context stays usable afterwards."""
import time

import pytest
import torch

from linear_attention_recurrence_gated_gb300 import gdn as G
from linear_attention_recurrence_gated_gb300 import workloads as W
import parity

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.time()
    assert G.gdn_debug_wait_timeout(ws) == G.GDN_OK
    assert G.gdn_check(ws) == 5          # GDN_ERR_TIMEOUT
    elapsed = time.time() - t0
    assert 1.5 < elapsed < 30.0, elapsed  # the wait gave up at its 2 s limit
    assert G.gdn_check(ws) == G.GDN_OK    # the check cleared the word
    # the context still runs a forward pass correctly
    w = W.custom(B=1, T=70, H=1, dk=64, dv=64, dtype="bf16", seed=31)
    inp = W.generate(w)
    ro, rs, _, _ = parity.compare(inp)
    to, ts = parity.TOL[torch.bfloat16]
    assert ro <= to and rs <= ts
