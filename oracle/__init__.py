"""Oracle for the gated delta rule forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls anything here, and this
package imports nothing from the product.

Contents
--------
``forward``      the token-by-token fp64 recurrence (C, ``gdn_oracle.c``):
                 S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
                 o_t = S_t q_t, alpha_t = exp(g_t) -- the gated delta rule of
                 Yang et al. (arXiv 2412.06464), named by "v1.0 Architecture &
                 Design Spec" section 2.3; loop structure after "Model
                 Architecture Walkthrough" section 5.5, Step 5.
``chunked``      an independent fp64 numpy statement of the chunked (WY/UT)
                 form, used only to pin the sequential oracle against it.
``diag``         the HyMo pages' own recurrence, per-state-row decay
                 exp(g_t A) with A = -exp(A_log), write key b, read key c
                 ("Model Architecture Walkthrough" section 5.2.1), token by
                 token in fp64 numpy; ``diag.forward_delta`` the same decay
                 combined with the delta rule's erase and beta.
``grad``         the backward pass (dq, dk, dv, dg, dbeta, d initial state):
                 torch.autograd over the fp64 token loop on the CPU.
``block``        the GDN block's prologue (causal depthwise conv1d + SiLU) and
                 epilogue ((o + D v) * g_gate), same page, sections 5.4-5.5.

Parity status of each function is recorded in its docstring; every function
here is pinned by a CPU test in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")

MODE_DELTA = 0  # gated delta rule (the method)
MODE_GLA = 1    # erase-off, beta-free scalar-decay recurrence (a pin only)

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` with gcc into ``oracle/_build``; return the path."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the C signature on a loaded oracle library (also used for test copies)."""
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gdn_oracle_forward.restype = ctypes.c_int
    lib.gdn_oracle_forward.argtypes = [
        dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_longlong),
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, dp, dp, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


def _as_f64(x) -> np.ndarray:
    """Exact upcast of stored values (fp32/bf16/fp64) to a C-contiguous fp64 array."""
    if hasattr(x, "detach"):  # a torch tensor: upcast through torch (bf16 has no numpy dtype)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def forward(q, k, v, g, beta, initial_state=None, cu_seqlens=None, *,
            mode: int = MODE_DELTA, qk_l2norm: bool = False,
            threads: int | None = None, return_final_state: bool = True):
    """Run the token-by-token fp64 oracle.

    Shapes follow the library's layout: q, k ``[B, T, H, dk]``; v ``[B, T, H, dv]``;
    g, beta ``[B, T, H]``; initial_state ``[N, H, dk, dv]`` (the transposed
    state H = S^T) or None for zeros.  With ``cu_seqlens`` (length N+1) B must be
    1 and sequence n is rows ``cu[n]:cu[n+1]``; without it the N = B rows of the
    batch are the sequences.  Inputs may be numpy arrays or torch tensors of any
    float dtype; they are upcast exactly to fp64.

    Returns ``(o, final_state)`` as fp64 numpy arrays, ``o`` shaped like v and
    ``final_state`` ``[N, H, dk, dv]`` (None when ``return_final_state`` is False).
    """
    q = _as_f64(q); k = _as_f64(k); v = _as_f64(v); g = _as_f64(g)
    if q.ndim != 4 or k.shape != q.shape or v.ndim != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("oracle: q,k must be [B,T,H,dk] and v [B,T,H,dv]")
    B, T, H, dk = q.shape
    dv = v.shape[3]
    if g.shape != (B, T, H):
        raise ValueError("oracle: g must be [B,T,H]")
    if mode == MODE_DELTA:
        beta = _as_f64(beta)
        if beta.shape != (B, T, H):
            raise ValueError("oracle: beta must be [B,T,H]")
    else:
        beta = np.zeros((B, T, H)) if beta is None else _as_f64(beta)
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("oracle: cu_seqlens needs B == 1")
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("oracle: cu_seqlens must rise from 0 to T")
    N = len(cu) - 1
    s0 = None
    if initial_state is not None:
        s0 = _as_f64(initial_state)
        if s0.shape != (N, H, dk, dv):
            raise ValueError("oracle: initial_state must be [N,H,dk,dv]")
    o = np.zeros((B, T, H, dv))
    sN = np.zeros((N, H, dk, dv)) if return_final_state else None

    lib = _load()
    dp = ctypes.POINTER(ctypes.c_double)

    def ptr(a):
        return None if a is None else a.ctypes.data_as(dp)

    rc = lib.gdn_oracle_forward(
        ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(s0),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        N, H, dk, dv, int(mode), int(bool(qk_l2norm)), ptr(o), ptr(sN),
        int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle: gdn_oracle_forward returned {rc}")
    return o, sN


from . import chunked  # noqa: E402  (numpy-only; no C build needed)

__all__ = ["forward", "build", "chunked", "default_threads", "MODE_DELTA", "MODE_GLA"]
