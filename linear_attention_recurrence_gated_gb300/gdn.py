"""Python binding of the C ABI in ``include/gdn.h`` (argument marshalling only).

Every function here has the name of the C entry point it calls.  The binding
checks tensor devices, dtypes, shapes and contiguity, passes raw device
pointers and the current CUDA stream, and turns status codes into
exceptions.  It computes nothing itself and has no fallback: if ``libgdn.so``
is missing or CUDA is unavailable it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK = 0
(GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA, GDN_ERR_TIMEOUT,
 GDN_ERR_BAD_SEQLENS, GDN_ERR_DEVICE_CHECK) = range(1, 8)
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_WORKSPACE", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_TIMEOUT",
                6: "GDN_ERR_BAD_SEQLENS", 7: "GDN_ERR_DEVICE_CHECK"}
GDN_F32, GDN_BF16 = 0, 1
GDN_QK_L2NORM = 1 << 0
GDN_FORCE_SIMT = 1 << 1
GDN_GATE_SIGMOID = 1 << 2
GDN_BETA_LOGITS = 1 << 3
GDN_DEBUG_CHECKS = 1 << 4
GDN_SEQ_SPLIT = 1 << 5
# site codes of a GDN_ERR_DEVICE_CHECK record (gdn_check_record)
DEBUG_SITES = {1: "q", 2: "k", 3: "v", 4: "g", 5: "beta", 6: "o", 7: "initial_state",
               8: "final_state", 9: "out_gate", 10: "tma_x"}
CHUNK_SIZE = 64

# Every symbol include/gdn.h declares.
EXPORTED = ("gdn_fwd_workspace_size", "gdn_workspace_init", "gdn_fwd", "gdn_check",
            "gdn_status_string", "gdn_fwd_kernel_name", "gdn_fwd_static_scratch",
            "gdn_decode", "gdn_diag_workspace_size", "gdn_diag_fwd", "gdn_conv_silu",
            "gdn_bwd_workspace_size", "gdn_bwd", "gdn_fwd_debug", "gdn_check_record",
            "gdn_fwd_kernel_name_chunk", "gdn_fwd_split_segments", "gdn_fwd_split_workspace_size",
            "gdn_diag_delta_workspace_size", "gdn_diag_delta_fwd")
# ... and include/gdn_debug.h (self-tests of the failure reporting).
DEBUG_EXPORTED = ("gdn_debug_wait_timeout",)

_lib = None
_lock = threading.Lock()


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """Load ``libgdn.so`` (raises if it was not built; there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} not found: build it with "
                    "`python -m linear_attention_recurrence_gated_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
            L.gdn_fwd_workspace_size.restype = sz
            L.gdn_fwd_workspace_size.argtypes = [i32, i32, i32, i32, u32]
            L.gdn_workspace_init.restype = ctypes.c_int
            L.gdn_workspace_init.argtypes = [vp, sz, vp]
            L.gdn_fwd.restype = ctypes.c_int
            L.gdn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                  i32, i32, i32, i32, i32, i32, i32, ctypes.c_int, u32,
                                  vp, sz, vp]
            L.gdn_check.restype = ctypes.c_int
            L.gdn_check.argtypes = [vp, vp]
            L.gdn_check_record.restype = ctypes.c_int
            L.gdn_check_record.argtypes = [vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                           ctypes.POINTER(i32)]
            L.gdn_fwd_debug.restype = ctypes.c_int
            L.gdn_fwd_debug.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                        i32, i32, i32, i32, i32, i32, i32, ctypes.c_int, u32,
                                        vp, sz, ctypes.POINTER(GdnExtents), vp]
            L.gdn_debug_wait_timeout.restype = ctypes.c_int
            L.gdn_debug_wait_timeout.argtypes = [vp, sz, vp]
            L.gdn_status_string.restype = ctypes.c_char_p
            L.gdn_status_string.argtypes = [i32]
            L.gdn_fwd_kernel_name.restype = ctypes.c_char_p
            L.gdn_fwd_kernel_name.argtypes = [i32, i32, ctypes.c_int, u32]
            L.gdn_fwd_kernel_name_chunk.restype = ctypes.c_char_p
            L.gdn_fwd_kernel_name_chunk.argtypes = [i32, i32, i32, ctypes.c_int, u32]
            L.gdn_fwd_split_workspace_size.restype = sz
            L.gdn_fwd_split_workspace_size.argtypes = [i32, i32, i32, i32, i32]
            L.gdn_fwd_split_segments.restype = i32
            L.gdn_fwd_split_segments.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_int, u32,
                                                 i32]
            L.gdn_fwd_static_scratch.restype = ctypes.c_int
            L.gdn_fwd_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 i32, i32, i32, i32, i32, i32, i32,
                                                 ctypes.c_int, u32, i32, vp]
            L.gdn_decode.restype = ctypes.c_int
            L.gdn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp,
                                     i32, i32, i32, i32, ctypes.c_int, u32, vp]
            L.gdn_bwd_workspace_size.restype = sz
            L.gdn_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32]
            L.gdn_bwd.restype = ctypes.c_int
            L.gdn_bwd.argtypes = [vp] * 15 + [i32] * 6 + [ctypes.c_int, u32, vp, sz, vp]
            L.gdn_conv_silu.restype = ctypes.c_int
            L.gdn_conv_silu.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int, vp]
            L.gdn_diag_workspace_size.restype = sz
            L.gdn_diag_workspace_size.argtypes = [i32, i32, i32, i32, i32]
            L.gdn_diag_fwd.restype = ctypes.c_int
            L.gdn_diag_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                       i32, i32, i32, i32, i32, ctypes.c_int, u32, vp, sz, vp]
            L.gdn_diag_delta_workspace_size.restype = sz
            L.gdn_diag_delta_workspace_size.argtypes = [i32, i32, i32, i32, i32]
            L.gdn_diag_delta_fwd.restype = ctypes.c_int
            L.gdn_diag_delta_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                             i32, i32, i32, i32, i32, ctypes.c_int, u32, vp, sz,
                                             vp]
            _lib = L
    return _lib


class GdnExtents(ctypes.Structure):
    """``gdn_extents``: elements each buffer of a forward call holds."""
    _fields_ = [(n, ctypes.c_int64) for n in ("q", "k", "v", "g", "beta", "o", "initial_state",
                                              "final_state", "out_gate")]


def status_string(status: int) -> str:
    try:
        return lib().gdn_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(int(status), f"status {status}")


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return GDN_F32
    if t == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"gdn: unsupported storage dtype {t} (float32 or bfloat16)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def gdn_fwd_workspace_size(num_seqs: int, num_heads: int, head_dim_k: int, head_dim_v: int,
                           flags: int = 0) -> int:
    return int(lib().gdn_fwd_workspace_size(num_seqs, num_heads, head_dim_k, head_dim_v, flags))


def gdn_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    st = lib().gdn_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_workspace_init")


def gdn_fwd_split_workspace_size(num_seqs: int, seq_len: int, num_heads: int, head_dim_k: int,
                                 head_dim_v: int) -> int:
    return int(lib().gdn_fwd_split_workspace_size(num_seqs, seq_len, num_heads, head_dim_k,
                                                  head_dim_v))


def new_workspace(num_seqs, num_heads, head_dim_k, head_dim_v, flags=0, device=None,
                  seq_len=None):
    """A zeroed workspace of the size gdn_fwd needs (the caller keeps it).
    With GDN_SEQ_SPLIT in ``flags`` pass ``seq_len`` (tokens per sequence of a
    dense call): a split call keeps per-token maps in the workspace."""
    if (flags & GDN_SEQ_SPLIT) and seq_len is not None:
        n = gdn_fwd_split_workspace_size(num_seqs, seq_len, num_heads, head_dim_k, head_dim_v)
    else:
        n = gdn_fwd_workspace_size(num_seqs, num_heads, head_dim_k, head_dim_v, flags)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def gdn_check(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(lib().gdn_check(_ptr(workspace), _stream_handle(stream)))


def gdn_check_record(workspace: torch.Tensor, stream=None):
    """gdn_check that also returns where the error arose:
    ``(status, seq, head, site)`` (site codes in ``DEBUG_SITES``)."""
    seq, head, site = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = lib().gdn_check_record(_ptr(workspace), _stream_handle(stream), ctypes.byref(seq),
                                ctypes.byref(head), ctypes.byref(site))
    return int(st), seq.value, head.value, site.value


def gdn_debug_wait_timeout(workspace: torch.Tensor, stream=None) -> int:
    """Enqueue the self-test whose bounded waits must give up (about 2 s) and
    report GDN_ERR_TIMEOUT in the workspace status word; returns the launch
    status (read the device status with gdn_check)."""
    return int(lib().gdn_debug_wait_timeout(_ptr(workspace),
                                            workspace.numel() * workspace.element_size(),
                                            _stream_handle(stream)))


def gdn_fwd_kernel_name(head_dim_k, head_dim_v, dtype: torch.dtype, flags: int = 0,
                        chunk_size: int = CHUNK_SIZE):
    r = lib().gdn_fwd_kernel_name_chunk(head_dim_k, head_dim_v, chunk_size, _dtype_code(dtype),
                                        flags)
    return None if r is None else r.decode()


def gdn_fwd_split_segments(num_seqs, seq_len, num_heads, head_dim_k, head_dim_v,
                           dtype: torch.dtype, flags: int = 0, chunk_size: int = CHUNK_SIZE,
                           varlen: bool = False) -> int:
    """Segments per sequence a gdn_fwd call with these sizes is cut into on the
    current device (1: not split, one kernel launch; >= 3: three launches);
    0 for sizes gdn_fwd rejects."""
    return int(lib().gdn_fwd_split_segments(num_seqs, seq_len, num_heads, head_dim_k,
                                            head_dim_v, chunk_size, _dtype_code(dtype), flags,
                                            1 if varlen else 0))


def _check_fwd_tensors(where, q, k, v, g, beta, initial_state, cu_seqlens, o, final_state,
                       D_skip=None, out_gate=None):
    """The tensor checks every forward entry point makes before it calls the
    library: device, contiguity, dtypes and shapes of inputs and of any output
    passed in.  Returns (N, H, dk, dv)."""
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError(f"{where}: q, k, v must be [B, T, H, D]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    tensors = [q, k, v, g, beta] + [t for t in (initial_state, cu_seqlens, o, final_state,
                                                D_skip, out_gate) if t is not None]
    for t in tensors:
        if not t.is_cuda:
            raise ValueError(f"{where}: every tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError(f"{where}: every tensor must be contiguous")
    _dtype_code(q.dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise TypeError(f"{where}: q, k, v and beta must share one storage dtype")
    if g.dtype != torch.float32:
        raise TypeError(f"{where}: g must be float32")
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or g.shape != (B, T, H) or \
            beta.shape != (B, T, H):
        raise ValueError(f"{where}: shape mismatch among q, k, v, g, beta")
    if initial_state is not None and (initial_state.dtype != torch.float32 or
                                      initial_state.shape != (N, H, dk, dv)):
        raise ValueError(f"{where}: initial_state must be float32 [N, H, dk, dv]")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError(f"{where}: cu_seqlens must be int32")
    if o is not None and (o.shape != v.shape or o.dtype != v.dtype):
        raise ValueError(f"{where}: o must match v in shape and dtype")
    if final_state is not None and (final_state.dtype != torch.float32 or
                                    final_state.shape != (N, H, dk, dv)):
        raise ValueError(f"{where}: final_state must be float32 [N, H, dk, dv]")
    if D_skip is not None and (D_skip.dtype != torch.float32 or tuple(D_skip.shape) != (H,)):
        raise ValueError(f"{where}: D_skip must be float32 [H]")
    if out_gate is not None and (out_gate.dtype != torch.float32 or out_gate.shape != (B, T, H)):
        raise ValueError(f"{where}: out_gate must be float32 [B, T, H]")
    return N, H, dk, dv


def _fwd_flags(qk_l2norm, beta_logits, force_simt, debug_checks, seq_split=False):
    return (GDN_QK_L2NORM if qk_l2norm else 0) | (GDN_FORCE_SIMT if force_simt else 0) | \
        (GDN_BETA_LOGITS if beta_logits else 0) | (GDN_DEBUG_CHECKS if debug_checks else 0) | \
        (GDN_SEQ_SPLIT if seq_split else 0)


def gdn_fwd(q, k, v, g, beta, initial_state=None, cu_seqlens=None, *, o=None,
            final_state=None, output_final_state=True, workspace=None, D_skip=None,
            out_gate=None, qk_l2norm=False, beta_logits=False, force_simt=False,
            chunk_size=CHUNK_SIZE, stream=None, check=False, debug_checks=False,
            seq_split=False):
    """Forward pass of the gated delta rule through the C ABI.

    q, k ``[B, T, H, dk]``; v ``[B, T, H, dv]``; g ``[B, T, H]`` fp32; beta
    ``[B, T, H]``; all CUDA, contiguous, q/k/v/beta/o in one storage dtype
    (float32 or bfloat16).  initial_state ``[N, H, dk, dv]`` fp32 or None;
    cu_seqlens int32 ``[N+1]`` on the device (then B must be 1) or None.
    ``o`` / ``final_state`` may be given to write into preallocated outputs
    (``final_state`` may be ``initial_state``).  ``chunk_size`` is 32, 64 (the
    default) or 128.  Returns ``(o, final_state)``.
    ``D_skip`` ``[H]`` and ``out_gate`` ``[B, T, H]`` (fp32, optional) fuse the
    block epilogue o <- (o + D_skip[h] v) * out_gate; ``beta_logits`` makes the
    kernel use sigmoid(beta); ``qk_l2norm`` normalises q and k in-kernel.
    ``debug_checks`` sets GDN_DEBUG_CHECKS (range checks before every access);
    ``seq_split`` sets GDN_SEQ_SPLIT (long dense sequences with head_dim_k 128
    cut into segments computed in parallel; a given ``workspace`` must be sized
    by ``gdn_fwd_split_workspace_size``, e.g. ``new_workspace(..., GDN_SEQ_SPLIT,
    seq_len=T)``).
    With ``check=True`` the call synchronises and raises on a device-side error.
    """
    N, H, dk, dv = _check_fwd_tensors("gdn_fwd", q, k, v, g, beta, initial_state, cu_seqlens,
                                      o, final_state, D_skip, out_gate)
    if o is None:
        o = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    B, T = q.shape[:2]
    dcode = _dtype_code(q.dtype)
    flags = _fwd_flags(qk_l2norm, beta_logits, force_simt, debug_checks, seq_split)
    if workspace is None:
        workspace = new_workspace(N, H, dk, dv, flags, device=q.device,
                                  seq_len=T if cu_seqlens is None else None)
    st = lib().gdn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                       _ptr(cu_seqlens), _ptr(o), _ptr(final_state), _ptr(D_skip),
                       _ptr(out_gate), B, T, H, dk, dv, N, chunk_size, dcode, flags, _ptr(workspace),
                       workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_fwd")
    if check:
        st = gdn_check(workspace, stream)
        if st != GDN_OK:
            raise GdnError(st, "gdn_fwd (device)")
    return o, final_state


def gdn_fwd_static_scratch(q, k, v, g, beta, initial_state, cu_seqlens, o, final_state, *,
                           D_skip=None, out_gate=None, qk_l2norm=False, beta_logits=False,
                           force_simt=False, check=True, stream=None,
                           debug_checks=False) -> int:
    """Forward pass for callers that cannot allocate device memory.

    Same tensors as ``gdn_fwd`` but every output must be passed in (this call
    allocates nothing, not even through torch) and there is no workspace: the
    library's own 256-byte device array holds the status record.  With
    ``check`` the call synchronises and returns the device status code; the
    status is returned, not raised, so the caller decides.
    """
    if o is None:
        raise ValueError("gdn_fwd_static_scratch: o must be passed in (the call allocates nothing)")
    N, H, dk, dv = _check_fwd_tensors("gdn_fwd_static_scratch", q, k, v, g, beta,
                                      initial_state, cu_seqlens, o, final_state, D_skip,
                                      out_gate)
    B, T = q.shape[:2]
    flags = _fwd_flags(qk_l2norm, beta_logits, force_simt, debug_checks)
    return int(lib().gdn_fwd_static_scratch(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens),
        _ptr(o), _ptr(final_state), _ptr(D_skip), _ptr(out_gate), B, T, H, dk, dv, N, CHUNK_SIZE,
        _dtype_code(q.dtype),
        flags, 1 if check else 0, _stream_handle(stream)))


def gdn_fwd_debug(q, k, v, g, beta, initial_state, cu_seqlens, o, final_state, workspace, *,
                  declared=None, D_skip=None, out_gate=None, qk_l2norm=False,
                  beta_logits=False, force_simt=False, chunk_size=CHUNK_SIZE, stream=None):
    """``gdn_fwd_debug``: the forward pass with GDN_DEBUG_CHECKS against
    declared extents.  ``declared`` maps buffer names (``GdnExtents`` fields)
    to element counts; missing names take the count of the tensor passed (0
    for None).  Outputs and workspace are passed in.  Returns the host status;
    read the device record with ``gdn_check_record``."""
    N, H, dk, dv = _check_fwd_tensors("gdn_fwd_debug", q, k, v, g, beta, initial_state,
                                      cu_seqlens, o, final_state, D_skip, out_gate)
    B, T = q.shape[:2]
    ext = None
    if declared is not None:
        have = dict(q=q, k=k, v=v, g=g, beta=beta, o=o, initial_state=initial_state,
                    final_state=final_state, out_gate=out_gate)
        unknown = set(declared) - set(have)
        if unknown:
            raise ValueError(f"gdn_fwd_debug: unknown extents {sorted(unknown)}")
        ext = GdnExtents(**{n: int(declared.get(n, 0 if t is None else t.numel()))
                            for n, t in have.items()})
    flags = _fwd_flags(qk_l2norm, beta_logits, force_simt, True)
    return int(lib().gdn_fwd_debug(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens),
        _ptr(o), _ptr(final_state), _ptr(D_skip), _ptr(out_gate), B, T, H, dk, dv, N,
        chunk_size, _dtype_code(q.dtype), flags, _ptr(workspace),
        workspace.numel() * workspace.element_size(),
        None if ext is None else ctypes.byref(ext), _stream_handle(stream)))


def gdn_decode(q, k, v, g, beta, state=None, *, o=None, state_out=None, qk_l2norm=False,
               stream=None):
    """One recurrent step per (sequence, head) through the C ABI.

    q, k ``[N, H, dk]``; v ``[N, H, dv]``; g ``[N, H]`` fp32; beta ``[N, H]``;
    q/k/v/beta/o in one storage dtype (float32 or bfloat16).  ``state``
    ``[N, H, dk, dv]`` fp32 or None (zeros).  ``state_out`` may be given
    (``state_out=state`` updates the state in place); otherwise a new tensor is
    returned.  Returns ``(o, state_out)``.
    """
    N, H, dk = q.shape
    dv = v.shape[-1]
    for t in [q, k, v, g, beta] + [t for t in (state, o, state_out) if t is not None]:
        if not t.is_cuda:
            raise ValueError("gdn_decode: every tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("gdn_decode: every tensor must be contiguous")
    dcode = _dtype_code(q.dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise TypeError("gdn_decode: q, k, v and beta must share one storage dtype")
    if g.dtype != torch.float32:
        raise TypeError("gdn_decode: g must be float32")
    if k.shape != q.shape or v.shape[:2] != (N, H) or g.shape != (N, H) or beta.shape != (N, H):
        raise ValueError("gdn_decode: shape mismatch among q, k, v, g, beta")
    for name, t in (("state", state), ("state_out", state_out)):
        if t is not None and (t.dtype != torch.float32 or t.shape != (N, H, dk, dv)):
            raise ValueError(f"gdn_decode: {name} must be float32 [N, H, dk, dv]")
    if o is None:
        o = torch.empty_like(v)
    elif o.shape != v.shape or o.dtype != v.dtype:
        raise ValueError("gdn_decode: o must match v in shape and dtype")
    if state_out is None:
        state_out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    st = lib().gdn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                          _ptr(state_out), _ptr(o), N, H, dk, dv, dcode,
                          GDN_QK_L2NORM if qk_l2norm else 0, _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_decode")
    return o, state_out


def gdn_diag_workspace_size(batch: int, seq_len: int, num_heads: int, d_state: int,
                            head_dim: int) -> int:
    return int(lib().gdn_diag_workspace_size(batch, seq_len, num_heads, d_state, head_dim))


def new_diag_workspace(batch, seq_len, num_heads, d_state, head_dim, device=None):
    """A zeroed workspace of the size gdn_diag_fwd needs (the caller keeps it)."""
    n = gdn_diag_workspace_size(batch, seq_len, num_heads, d_state, head_dim)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def gdn_diag_fwd(v, b, c, g, A_log, initial_state=None, *, D_skip=None, out_gate=None,
                 gate_sigmoid=False, o=None, final_state=None, output_final_state=True,
                 workspace=None, stream=None, check=False):
    """The pages' diagonal-decay recurrence through the C ABI.

    v ``[B, T, H, D]``; b, c ``[B, T, H, S]`` (v, b, c and o in one storage
    dtype, float32 or bfloat16); g ``[B, T, H]`` fp32; A_log ``[H, S]`` fp32;
    initial_state ``[B, H, S, D]`` fp32 or None.  ``D_skip`` ``[H]`` and
    ``out_gate`` ``[B, T, H]`` (fp32) fuse the block epilogue
    o <- (o + D_skip v) * out_gate; ``gate_sigmoid`` makes g the logits of the
    decay gate (g = sigmoid(g) in the kernel).  Returns ``(o, final_state)``
    (``final_state`` None when ``output_final_state`` is False and none is given).
    A workspace made by ``new_diag_workspace`` for the same sizes may be reused
    across calls on one stream.
    """
    B, T, H, D = v.shape
    S = b.shape[-1]
    for t in [v, b, c, g, A_log] + [t for t in (initial_state, o, final_state, D_skip, out_gate)
                                    if t is not None]:
        if not t.is_cuda:
            raise ValueError("gdn_diag_fwd: every tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("gdn_diag_fwd: every tensor must be contiguous")
    dcode = _dtype_code(v.dtype)
    if b.dtype != v.dtype or c.dtype != v.dtype:
        raise TypeError("gdn_diag_fwd: v, b and c must share one storage dtype")
    if g.dtype != torch.float32 or A_log.dtype != torch.float32:
        raise TypeError("gdn_diag_fwd: g and A_log must be float32")
    if b.shape != (B, T, H, S) or c.shape != (B, T, H, S) or g.shape != (B, T, H) or \
            A_log.shape != (H, S):
        raise ValueError("gdn_diag_fwd: shape mismatch among v, b, c, g, A_log")
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is not None and (t.dtype != torch.float32 or t.shape != (B, H, S, D)):
            raise ValueError(f"gdn_diag_fwd: {name} must be float32 [B, H, S, D]")
    if D_skip is not None and (D_skip.dtype != torch.float32 or D_skip.shape != (H,)):
        raise ValueError("gdn_diag_fwd: D_skip must be float32 [H]")
    if out_gate is not None and (out_gate.dtype != torch.float32 or out_gate.shape != (B, T, H)):
        raise ValueError("gdn_diag_fwd: out_gate must be float32 [B, T, H]")
    if o is None:
        o = torch.empty_like(v)
    elif o.shape != v.shape or o.dtype != v.dtype:
        raise ValueError("gdn_diag_fwd: o must match v in shape and dtype")
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, S, D), dtype=torch.float32, device=v.device)
    if workspace is None:
        workspace = new_diag_workspace(B, T, H, S, D, device=v.device)
    st = lib().gdn_diag_fwd(_ptr(v), _ptr(b), _ptr(c), _ptr(g), _ptr(A_log), _ptr(D_skip),
                            _ptr(out_gate), _ptr(initial_state), _ptr(o), _ptr(final_state),
                            B, T, H, S, D, dcode, GDN_GATE_SIGMOID if gate_sigmoid else 0,
                            _ptr(workspace),
                            workspace.numel() * workspace.element_size(),
                            _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_diag_fwd")
    if check:
        st = gdn_check(workspace, stream)
        if st != GDN_OK:
            raise GdnError(st, "gdn_diag_fwd (device)")
    return o, final_state


def gdn_diag_delta_workspace_size(batch: int, seq_len: int, num_heads: int, d_state: int,
                                  head_dim: int) -> int:
    return int(lib().gdn_diag_delta_workspace_size(batch, seq_len, num_heads, d_state,
                                                   head_dim))


def new_diag_delta_workspace(batch, seq_len, num_heads, d_state, head_dim, device=None):
    """A zeroed workspace of the size gdn_diag_delta_fwd needs (the caller keeps it)."""
    n = gdn_diag_delta_workspace_size(batch, seq_len, num_heads, d_state, head_dim)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def gdn_diag_delta_fwd(v, b, c, g, A_log, beta, initial_state=None, *, D_skip=None,
                       out_gate=None, gate_sigmoid=False, beta_logits=False, o=None,
                       final_state=None, output_final_state=True, workspace=None, stream=None,
                       check=False):
    """The pages' diagonal decay combined with the delta rule, through the C ABI.

    Tensors as ``gdn_diag_fwd`` plus beta ``[B, T, H]`` in the storage dtype of
    v, b, c.  ``beta_logits`` makes beta the logits of the write strength
    (sigmoid in the kernel).  Returns ``(o, final_state)``.  A workspace made by
    ``new_diag_delta_workspace`` for the same sizes may be reused across calls
    on one stream.
    """
    B, T, H, D = v.shape
    S = b.shape[-1]
    for t in [v, b, c, g, A_log, beta] + [t for t in (initial_state, o, final_state, D_skip,
                                                      out_gate) if t is not None]:
        if not t.is_cuda:
            raise ValueError("gdn_diag_delta_fwd: every tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("gdn_diag_delta_fwd: every tensor must be contiguous")
    dcode = _dtype_code(v.dtype)
    if b.dtype != v.dtype or c.dtype != v.dtype or beta.dtype != v.dtype:
        raise TypeError("gdn_diag_delta_fwd: v, b, c and beta must share one storage dtype")
    if g.dtype != torch.float32 or A_log.dtype != torch.float32:
        raise TypeError("gdn_diag_delta_fwd: g and A_log must be float32")
    if b.shape != (B, T, H, S) or c.shape != (B, T, H, S) or g.shape != (B, T, H) or \
            beta.shape != (B, T, H) or A_log.shape != (H, S):
        raise ValueError("gdn_diag_delta_fwd: shape mismatch among v, b, c, g, beta, A_log")
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is not None and (t.dtype != torch.float32 or t.shape != (B, H, S, D)):
            raise ValueError(f"gdn_diag_delta_fwd: {name} must be float32 [B, H, S, D]")
    if D_skip is not None and (D_skip.dtype != torch.float32 or D_skip.shape != (H,)):
        raise ValueError("gdn_diag_delta_fwd: D_skip must be float32 [H]")
    if out_gate is not None and (out_gate.dtype != torch.float32 or out_gate.shape != (B, T, H)):
        raise ValueError("gdn_diag_delta_fwd: out_gate must be float32 [B, T, H]")
    if o is None:
        o = torch.empty_like(v)
    elif o.shape != v.shape or o.dtype != v.dtype:
        raise ValueError("gdn_diag_delta_fwd: o must match v in shape and dtype")
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, S, D), dtype=torch.float32, device=v.device)
    if workspace is None:
        workspace = new_diag_delta_workspace(B, T, H, S, D, device=v.device)
    flags = (GDN_GATE_SIGMOID if gate_sigmoid else 0) | (GDN_BETA_LOGITS if beta_logits else 0)
    st = lib().gdn_diag_delta_fwd(_ptr(v), _ptr(b), _ptr(c), _ptr(g), _ptr(A_log), _ptr(beta),
                                  _ptr(D_skip), _ptr(out_gate), _ptr(initial_state), _ptr(o),
                                  _ptr(final_state), B, T, H, S, D, dcode, flags,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_diag_delta_fwd")
    if check:
        st = gdn_check(workspace, stream)
        if st != GDN_OK:
            raise GdnError(st, "gdn_diag_delta_fwd (device)")
    return o, final_state


def gdn_conv_silu(x, w, x_prev=None, *, y=None, x_tail=None, stream=None):
    """Causal depthwise conv1d + SiLU through the C ABI (the GDN block prologue).

    x ``[B, T, C]`` (float32 or bfloat16); w ``[C, K]`` fp32 (PyTorch's Conv1d
    weight ``[C, 1, K]`` squeezed); x_prev ``[B, K-1, C]`` or None (zeros).
    ``x_tail`` (``[B, K-1, C]``, x's dtype) receives the last K-1 inputs when
    given.  Returns ``y``.
    """
    B, T, C = x.shape
    K = w.shape[-1]
    for t in [x, w] + [t for t in (x_prev, y, x_tail) if t is not None]:
        if not t.is_cuda:
            raise ValueError("gdn_conv_silu: every tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("gdn_conv_silu: every tensor must be contiguous")
    dcode = _dtype_code(x.dtype)
    if w.dtype != torch.float32 or w.shape != (C, K):
        raise ValueError("gdn_conv_silu: w must be float32 [C, K]")
    for name, t in (("x_prev", x_prev), ("x_tail", x_tail)):
        if t is not None and (t.dtype != x.dtype or t.shape != (B, K - 1, C)):
            raise ValueError(f"gdn_conv_silu: {name} must be [B, K-1, C] in x's dtype")
    if y is None:
        y = torch.empty_like(x)
    elif y.shape != x.shape or y.dtype != x.dtype:
        raise ValueError("gdn_conv_silu: y must match x")
    st = lib().gdn_conv_silu(_ptr(x), _ptr(w), _ptr(x_prev), _ptr(y), _ptr(x_tail), B, T, C, K,
                             dcode, _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_conv_silu")
    return y


def gdn_bwd_workspace_size(num_seqs: int, seq_len: int, num_heads: int, head_dim_k: int,
                           head_dim_v: int) -> int:
    return int(lib().gdn_bwd_workspace_size(num_seqs, seq_len, num_heads, head_dim_k, head_dim_v))


def gdn_bwd(q, k, v, g, beta, d_o, initial_state=None, cu_seqlens=None, d_final_state=None, *,
            grads=None, workspace=None, stream=None, check=False):
    """Backward pass of ``gdn_fwd`` through the C ABI.

    Inputs as ``gdn_fwd`` plus ``d_o`` (like v) and ``d_final_state``
    (``[N, H, dk, dv]`` fp32 or None).  Returns a dict of fp32 tensors
    ``dq, dk, dv, dg, dbeta, dh0`` (``grads`` may supply them preallocated).
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    for t in [q, k, v, g, beta, d_o] + [t for t in (initial_state, cu_seqlens, d_final_state)
                                        if t is not None]:
        if not t.is_cuda:
            raise ValueError("gdn_bwd: every tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("gdn_bwd: every tensor must be contiguous")
    dcode = _dtype_code(q.dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype or d_o.dtype != q.dtype:
        raise TypeError("gdn_bwd: q, k, v, beta and d_o must share one storage dtype")
    if g.dtype != torch.float32:
        raise TypeError("gdn_bwd: g must be float32")
    if d_o.shape != v.shape:
        raise ValueError("gdn_bwd: d_o must match v")
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None and (t.dtype != torch.float32 or t.shape != (N, H, dk, dv)):
            raise ValueError(f"gdn_bwd: {name} must be float32 [N, H, dk, dv]")
    f32 = dict(dtype=torch.float32, device=q.device)
    if grads is None:
        grads = {"dq": torch.empty((B, T, H, dk), **f32), "dk": torch.empty((B, T, H, dk), **f32),
                 "dv": torch.empty((B, T, H, dv), **f32), "dg": torch.empty((B, T, H), **f32),
                 "dbeta": torch.empty((B, T, H), **f32),
                 "dh0": torch.empty((N, H, dk, dv), **f32)}
    if workspace is None:
        n = gdn_bwd_workspace_size(N, T, H, dk, dv)
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    st = lib().gdn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                       _ptr(cu_seqlens), _ptr(d_o), _ptr(d_final_state), _ptr(grads["dq"]),
                       _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dg"]),
                       _ptr(grads["dbeta"]), _ptr(grads.get("dh0")), B, T, H, dk, dv, N, dcode,
                       0, _ptr(workspace), workspace.numel() * workspace.element_size(),
                       _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_bwd")
    if check:
        st = gdn_check(workspace, stream)
        if st != GDN_OK:
            raise GdnError(st, "gdn_bwd (device)")
    return grads
