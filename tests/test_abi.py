"""CPU tests of the C-ABI library: it loads, exports every symbol that
include/gdn.h declares, and rejects malformed calls on the host before
touching the GPU (no call here launches anything)."""
import ctypes
import os
import re

import pytest

from linear_attention_recurrence_gated_gb300 import build as gbuild
from linear_attention_recurrence_gated_gb300 import gdn as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return G.lib()


def declared_functions():
    hdr = open(os.path.join(ROOT, "include", "gdn.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", hdr)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(G.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_debug_header_symbols_are_exported(L):
    hdr = open(os.path.join(ROOT, "include", "gdn_debug.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    names = sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", hdr)))
    assert names == sorted(G.DEBUG_EXPORTED)
    for name in names:
        assert hasattr(L, name), name


def test_debug_wait_timeout_validates_on_host(L):
    vp = ctypes.c_void_p
    assert L.gdn_debug_wait_timeout(vp(None), 256, vp(0)) == 3
    assert L.gdn_debug_wait_timeout(vp(1 << 40), 255, vp(0)) == 3
    assert L.gdn_debug_wait_timeout(vp((1 << 40) + 8), 256, vp(0)) == 1


def test_status_strings(L):
    for code, name in G.STATUS_NAMES.items():
        assert G.status_string(code).startswith(name)
    assert G.status_string(99) == "GDN_ERR_UNKNOWN"


def test_workspace_size(L):
    assert G.gdn_fwd_workspace_size(8, 16, 64, 64) >= 256
    # GDN_SEQ_SPLIT with head_dim_k 128: 8 segments' states, X (dk x dv) and M (dk x dk)
    seg = 256 + 4 * 1 * 8 * 16 * 128 * (2 * 128 + 128)
    assert G.gdn_fwd_workspace_size(1, 16, 128, 128, G.GDN_SEQ_SPLIT) == seg
    assert G.gdn_fwd_workspace_size(1, 16, 64, 64, G.GDN_SEQ_SPLIT) == 256
    # ... and for a split call the per-token maps r, bf16 [tokens][heads][dk], 256-aligned
    assert G.gdn_fwd_split_workspace_size(1, 65536, 16, 128, 128) == \
        (seg + 255) // 256 * 256 + 2 * 65536 * 16 * 128
    assert G.gdn_fwd_split_workspace_size(1, 1000, 2, 64, 64) == 256
    assert G.gdn_fwd_split_workspace_size(0, 1000, 2, 128, 128) == 0
    assert G.gdn_fwd_workspace_size(0, 16, 64, 64) == 0


def test_split_segments_host_rules(L):
    """The split query's host-side rules (no device attribute is read on these
    paths): rejected sizes give 0; no GDN_SEQ_SPLIT, fp32 storage, other chunk
    sizes or head_dim_k 64 give 1 (never split)."""
    import torch
    S = G.gdn_fwd_split_segments
    assert S(0, 65536, 16, 128, 128, torch.bfloat16, G.GDN_SEQ_SPLIT) == 0
    assert S(1, 65536, 16, 48, 128, torch.bfloat16, G.GDN_SEQ_SPLIT) == 0
    assert S(1, 65536, 16, 128, 100, torch.bfloat16, G.GDN_SEQ_SPLIT) == 0
    assert S(1, 65536, 16, 128, 128, torch.bfloat16, 0) == 1
    assert S(1, 65536, 16, 128, 128, torch.float32, G.GDN_SEQ_SPLIT) == 1
    assert S(1, 65536, 16, 128, 128, torch.bfloat16, G.GDN_SEQ_SPLIT, chunk_size=32) == 1
    assert S(1, 65536, 16, 64, 128, torch.bfloat16, G.GDN_SEQ_SPLIT) == 1
    # debug calls run unsplit (the split's extra kernels check no declared extents)
    assert S(1, 65536, 16, 128, 128, torch.bfloat16, G.GDN_SEQ_SPLIT | G.GDN_DEBUG_CHECKS) == 1


def test_kernel_names(L):
    import torch
    assert G.gdn_fwd_kernel_name(64, 64, torch.float32) == "simt_fp32"
    assert G.gdn_fwd_kernel_name(48, 64, torch.bfloat16) is None
    assert G.gdn_fwd_kernel_name(64, 48, torch.bfloat16) is None
    # bf16 storage: tensor-core kernels where the head sizes allow, else the fp32 kernel
    assert G.gdn_fwd_kernel_name(64, 64, torch.bfloat16) == "tc64_bf16"
    assert G.gdn_fwd_kernel_name(64, 128, torch.bfloat16) == "tc64_bf16"
    assert G.gdn_fwd_kernel_name(128, 128, torch.bfloat16) == "tc128_bf16"
    assert G.gdn_fwd_kernel_name(32, 64, torch.bfloat16) == "simt_bf16"
    assert G.gdn_fwd_kernel_name(64, 96, torch.bfloat16) == "simt_bf16"
    assert G.gdn_fwd_kernel_name(64, 64, torch.bfloat16, G.GDN_QK_L2NORM) == "tc64_bf16"
    assert G.gdn_fwd_kernel_name(128, 128, torch.bfloat16, G.GDN_QK_L2NORM) == "tc128_bf16"
    assert G.gdn_fwd_kernel_name(64, 64, torch.bfloat16, G.GDN_FORCE_SIMT) == "simt_bf16"
    # chunk sizes 32 and 128: tensor-core variants for bf16 with head_dim_k 64
    assert G.gdn_fwd_kernel_name(64, 64, torch.bfloat16, chunk_size=32) == "tcc32_bf16"
    assert G.gdn_fwd_kernel_name(64, 128, torch.bfloat16, chunk_size=128) == "tcc128_bf16"
    assert G.gdn_fwd_kernel_name(64, 64, torch.bfloat16, G.GDN_QK_L2NORM, chunk_size=32) == "tcc32_bf16"
    assert G.gdn_fwd_kernel_name(128, 128, torch.bfloat16, chunk_size=32) == "simt_bf16"
    assert G.gdn_fwd_kernel_name(64, 96, torch.bfloat16, chunk_size=128) == "simt_bf16"
    assert G.gdn_fwd_kernel_name(64, 64, torch.float32, chunk_size=32) == "simt_fp32"
    assert G.gdn_fwd_kernel_name(64, 64, torch.bfloat16, G.GDN_FORCE_SIMT, chunk_size=128) == "simt_bf16"
    assert G.gdn_fwd_kernel_name(64, 64, torch.bfloat16, chunk_size=16) is None
    assert G.gdn_fwd_kernel_name(128, 128, torch.bfloat16, chunk_size=128) is None


# ---- host-side validation with fake (never dereferenced) device addresses ----
BASE = 1 << 40


def call(L, **over):
    B, T, H, dk, dv = 2, 100, 3, 64, 64
    rows = B * T * H
    a = dict(q=BASE, k=BASE + (1 << 30), v=BASE + (2 << 30), g=BASE + (3 << 30),
             beta=BASE + (4 << 30), s0=None, cu=None, o=BASE + (5 << 30),
             sN=BASE + (6 << 30), dskip=None, ogate=None, B=B, T=T, H=H, dk=dk, dv=dv, N=B,
             chunk=64, dtype=G.GDN_BF16, flags=0, ws=BASE + (7 << 30), ws_bytes=256)
    a.update(over)
    vp = ctypes.c_void_p
    return L.gdn_fwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]),
                     vp(a["s0"]), vp(a["cu"]), vp(a["o"]), vp(a["sN"]), vp(a["dskip"]),
                     vp(a["ogate"]), a["B"], a["T"],
                     a["H"], a["dk"], a["dv"], a["N"], a["chunk"], a["dtype"], a["flags"],
                     vp(a["ws"]), a["ws_bytes"], vp(0))


@pytest.mark.parametrize("over,code", [
    (dict(dk=48), 2), (dict(dk=256), 2), (dict(dv=48), 2), (dict(dv=288), 2),
    (dict(chunk=16), 2), (dict(chunk=256), 2), (dict(chunk=128, dk=128, dv=128), 2),
    (dict(dtype=7), 1), (dict(flags=1 << 9), 1),
    (dict(q=None), 1), (dict(o=None), 1), (dict(g=None), 1), (dict(beta=None), 1),
    (dict(q=BASE + 8), 1), (dict(o=BASE + (5 << 30) + 4), 1), (dict(sN=BASE + (6 << 30) + 2), 1),
    (dict(ws=None), 3), (dict(ws_bytes=255), 3), (dict(ws=BASE + (7 << 30) + 8), 1),
    (dict(B=0), 1), (dict(T=-1), 1), (dict(H=0), 1), (dict(N=3), 1),
    (dict(T=0, sN=None), 0),                               # no tokens, no state: nothing to do
    (dict(cu=BASE + (8 << 30)), 1),                        # cu_seqlens needs batch == 1
    (dict(B=1, N=70000, cu=BASE + (8 << 30)), 2),          # too many sequences
    (dict(o=BASE), 1),                                     # o aliases q
    (dict(o=BASE + (2 << 30) + 64), 1),                    # o overlaps v
    (dict(sN=BASE + (4 << 30)), 1),                        # final_state aliases beta
    (dict(s0=BASE + (6 << 30) + 16), 1),                   # initial/final partial overlap
    (dict(ws=BASE + (5 << 30)), 1),                        # workspace inside o
    (dict(ogate=BASE + (5 << 30)), 1),                     # out_gate inside o
    (dict(dskip=BASE + (6 << 30) + 32), 1),                # D_skip inside final_state
    (dict(ogate=BASE + (9 << 30) + 4), 1),                 # out_gate misaligned
    (dict(flags=G.GDN_GATE_SIGMOID), 1),                   # a gdn_diag_fwd flag
])
def test_host_validation_rejects_before_launch(L, over, code):
    assert call(L, **over) == code


def call_debug(L, declared, **over):
    """gdn_fwd_debug with the fake addresses of `call` and declared extents
    (None = from the shapes)."""
    B, T, H, dk, dv = 2, 100, 3, 64, 64
    a = dict(q=BASE, k=BASE + (1 << 30), v=BASE + (2 << 30), g=BASE + (3 << 30),
             beta=BASE + (4 << 30), s0=None, cu=None, o=BASE + (5 << 30),
             sN=BASE + (6 << 30), B=B, T=T, H=H, dk=dk, dv=dv, N=B, flags=0,
             ws=BASE + (7 << 30), ws_bytes=256)
    a.update(over)
    vp = ctypes.c_void_p
    ext = None if declared is None else ctypes.byref(G.GdnExtents(**declared))
    return L.gdn_fwd_debug(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]),
                           vp(a["s0"]), vp(a["cu"]), vp(a["o"]), vp(a["sN"]), vp(None),
                           vp(None), a["B"], a["T"], a["H"], a["dk"], a["dv"], a["N"], 64,
                           G.GDN_BF16, a["flags"], vp(a["ws"]), a["ws_bytes"], ext, vp(0))


FULL = dict(q=2 * 100 * 3 * 64, k=2 * 100 * 3 * 64, v=2 * 100 * 3 * 64, g=600, beta=600,
            o=2 * 100 * 3 * 64, initial_state=2 * 3 * 64 * 64, final_state=2 * 3 * 64 * 64,
            out_gate=600)


def test_debug_flag_and_extents_layout():
    assert G.GDN_DEBUG_CHECKS == 1 << 4
    hdr = open(os.path.join(ROOT, "include", "gdn.h")).read()
    assert "GDN_DEBUG_CHECKS = 1u << 4" in hdr
    fields = re.search(r"typedef struct gdn_extents \{(.*?)\} gdn_extents;", hdr, re.S).group(1)
    names = re.findall(r"\b([a-z_]+)\s*[,;]", fields)
    assert names == [n for n, _ in G.GdnExtents._fields_]
    assert ctypes.sizeof(G.GdnExtents) == 8 * len(names)


@pytest.mark.parametrize("declared,over,code", [
    (dict(FULL, q=-1), {}, 1),                        # a negative extent
    (dict(FULL, out_gate=-5), {}, 1),                 # even for a NULL buffer
    (FULL, dict(dk=48), 2),                           # gdn_fwd's own validation first
    (FULL, dict(ws=None), 3),
    (FULL, dict(flags=1 << 9), 1),
    (dict(FULL, final_state=10), dict(T=0), 1),       # no tokens: the state copy is checked here
    (dict(FULL, initial_state=10), dict(T=0, s0=BASE + (8 << 30)), 1),
    (dict(FULL, final_state=10), dict(T=0, sN=None), 0),  # nothing to copy
])
def test_fwd_debug_validates_on_host(L, declared, over, code):
    assert call_debug(L, declared, **over) == code


def test_debug_flag_accepted_by_validation(L):
    # the flag passes gdn_fwd's mask: a malformed call still fails for its real reason
    assert call(L, flags=G.GDN_DEBUG_CHECKS, dk=48) == 2
    assert call(L, flags=G.GDN_DEBUG_CHECKS, T=0, sN=None) == 0


def test_check_record_null_workspace(L):
    seq, head, site = ctypes.c_int32(5), ctypes.c_int32(5), ctypes.c_int32(5)
    assert L.gdn_check_record(None, ctypes.c_void_p(0), ctypes.byref(seq), ctypes.byref(head),
                              ctypes.byref(site)) == 3
    assert (seq.value, head.value, site.value) == (-1, -1, 0)


def test_workspace_init_rejects_small(L):
    assert L.gdn_workspace_init(ctypes.c_void_p(BASE), 16, ctypes.c_void_p(0)) == 3
    assert L.gdn_workspace_init(None, 4096, ctypes.c_void_p(0)) == 3


def test_check_rejects_null_workspace(L):
    assert L.gdn_check(None, ctypes.c_void_p(0)) == 3


def call_decode(L, **over):
    N, H, dk, dv = 4, 3, 64, 64
    a = dict(q=BASE, k=BASE + (1 << 30), v=BASE + (2 << 30), g=BASE + (3 << 30),
             beta=BASE + (4 << 30), s_in=BASE + (6 << 30), s_out=BASE + (6 << 30),
             o=BASE + (5 << 30), N=N, H=H, dk=dk, dv=dv, dtype=G.GDN_BF16, flags=0)
    a.update(over)
    vp = ctypes.c_void_p
    return L.gdn_decode(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]),
                        vp(a["s_in"]), vp(a["s_out"]), vp(a["o"]), a["N"], a["H"], a["dk"],
                        a["dv"], a["dtype"], a["flags"], vp(0))


@pytest.mark.parametrize("over,code", [
    (dict(dk=48), 2), (dict(dk=256), 2), (dict(dv=48), 2), (dict(dv=288), 2),
    (dict(dtype=7), 1), (dict(flags=G.GDN_FORCE_SIMT), 1), (dict(flags=1 << 9), 1),
    (dict(q=None), 1), (dict(o=None), 1), (dict(s_out=None), 1), (dict(g=None), 1),
    (dict(q=BASE + 8), 1), (dict(s_out=BASE + (6 << 30) + 4, s_in=None), 1),
    (dict(N=0), 1), (dict(H=0), 1), (dict(N=70000), 2),
    (dict(o=BASE), 1),                                      # o aliases q
    (dict(s_out=BASE + (2 << 30)), 1),                      # state_out aliases v
    (dict(s_in=BASE + (6 << 30) + 16), 1),                  # state in/out partial overlap
    (dict(o=BASE + (6 << 30) + 64), 1),                     # o inside the state
])
def test_decode_host_validation_rejects_before_launch(L, over, code):
    assert call_decode(L, **over) == code


# ---- gdn_diag_fwd (the pages' diagonal-decay recurrence) ----
def test_diag_workspace_size(L):
    # 4 x 40 heads x 32 blocks of 128 tokens: a flag, an aggregate map and an end state each
    n = G.gdn_diag_workspace_size(4, 4096, 40, 32, 32)
    tasks = 4 * 40 * 32
    assert n >= 256 + tasks * (4 + (32 * 32 + 32) * 4 + 32 * 32 * 4)
    assert G.gdn_diag_workspace_size(1, 1, 1, 32, 32) > 256
    assert G.gdn_diag_workspace_size(0, 1, 1, 32, 32) == 0
    assert G.gdn_diag_workspace_size(1, 0, 1, 32, 32) == 0


def call_diag(L, **over):
    B, T, H, S, D = 2, 300, 3, 32, 32
    ws_need = G.gdn_diag_workspace_size(B, T, H, S, D)
    a = dict(v=BASE, b=BASE + (1 << 30), c=BASE + (2 << 30), g=BASE + (3 << 30),
             A=BASE + (4 << 30), Dk=None, og=None, s0=None, o=BASE + (5 << 30),
             sN=BASE + (6 << 30),
             B=B, T=T, H=H, S=S, D=D, dtype=G.GDN_BF16, flags=0, ws=BASE + (7 << 30),
             ws_bytes=ws_need)
    a.update(over)
    vp = ctypes.c_void_p
    return L.gdn_diag_fwd(vp(a["v"]), vp(a["b"]), vp(a["c"]), vp(a["g"]), vp(a["A"]),
                          vp(a["Dk"]), vp(a["og"]), vp(a["s0"]), vp(a["o"]), vp(a["sN"]),
                          a["B"], a["T"], a["H"], a["S"],
                          a["D"], a["dtype"], a["flags"], vp(a["ws"]), a["ws_bytes"], vp(0))


@pytest.mark.parametrize("over,code", [
    (dict(S=16), 2), (dict(D=64), 2), (dict(S=0), 1), (dict(D=-1), 1),
    (dict(B=0), 1), (dict(T=0), 1), (dict(H=0), 1),
    (dict(dtype=5), 1), (dict(flags=1), 1), (dict(flags=G.GDN_FORCE_SIMT), 1),
    (dict(Dk=BASE + (4 << 30) + 8), 1),                      # misaligned D_skip
    (dict(og=BASE + (5 << 30)), 1),                          # out_gate aliases o
    (dict(Dk=BASE + (6 << 30)), 1),                          # D_skip inside the final state
    (dict(v=None), 1), (dict(b=None), 1), (dict(c=None), 1), (dict(g=None), 1),
    (dict(A=None), 1), (dict(o=None), 1),
    (dict(c=BASE + (2 << 30) + 4), 1), (dict(sN=BASE + (6 << 30) + 8), 1),
    (dict(ws=None), 3), (dict(ws_bytes=256), 3), (dict(ws=BASE + (7 << 30) + 2), 1),
    (dict(o=BASE + (1 << 30)), 1),                           # o aliases b
    (dict(sN=BASE + (3 << 30)), 1),                          # final state aliases g
    (dict(s0=BASE + (5 << 30) + 1024), 1),                   # initial state inside o
    (dict(s0=BASE + (6 << 30) + 16), 1),                     # state in/out partial overlap
    (dict(sN=BASE + (7 << 30) + 4096), 1),                   # final state inside the workspace
    (dict(B=1 << 16, H=1 << 16), 2),                         # too many blocks
])
def test_diag_host_validation_rejects_before_launch(L, over, code):
    assert call_diag(L, **over) == code


# ---- gdn_diag_delta_fwd (diagonal decay combined with the delta rule) ----
def test_diag_delta_workspace_size(L):
    # 4 x 40 heads x 32 segments of 128 tokens: a flag and an end state each
    n = G.gdn_diag_delta_workspace_size(4, 4096, 40, 32, 32)
    tasks = 4 * 40 * 32
    assert n >= 256 + tasks * (4 + 32 * 32 * 4)
    assert G.gdn_diag_delta_workspace_size(1, 1, 1, 32, 32) > 256
    assert G.gdn_diag_delta_workspace_size(0, 1, 1, 32, 32) == 0
    assert G.gdn_diag_delta_workspace_size(1, 0, 1, 32, 32) == 0


def call_diag_delta(L, **over):
    B, T, H, S, D = 2, 300, 3, 32, 32
    ws_need = G.gdn_diag_delta_workspace_size(B, T, H, S, D)
    a = dict(v=BASE, b=BASE + (1 << 30), c=BASE + (2 << 30), g=BASE + (3 << 30),
             A=BASE + (4 << 30), beta=BASE + (8 << 30), Dk=None, og=None, s0=None,
             o=BASE + (5 << 30), sN=BASE + (6 << 30),
             B=B, T=T, H=H, S=S, D=D, dtype=G.GDN_BF16, flags=0, ws=BASE + (7 << 30),
             ws_bytes=ws_need)
    a.update(over)
    vp = ctypes.c_void_p
    return L.gdn_diag_delta_fwd(vp(a["v"]), vp(a["b"]), vp(a["c"]), vp(a["g"]), vp(a["A"]),
                                vp(a["beta"]), vp(a["Dk"]), vp(a["og"]), vp(a["s0"]),
                                vp(a["o"]), vp(a["sN"]), a["B"], a["T"], a["H"], a["S"],
                                a["D"], a["dtype"], a["flags"], vp(a["ws"]), a["ws_bytes"],
                                vp(0))


@pytest.mark.parametrize("over,code", [
    (dict(S=16), 2), (dict(D=64), 2), (dict(S=0), 1), (dict(B=0), 1), (dict(T=0), 1),
    (dict(dtype=5), 1), (dict(flags=1), 1), (dict(flags=G.GDN_QK_L2NORM), 1),
    (dict(beta=None), 1), (dict(v=None), 1), (dict(A=None), 1), (dict(o=None), 1),
    (dict(beta=BASE + (8 << 30) + 2), 1),                   # misaligned beta
    (dict(o=BASE + (8 << 30)), 1),                          # o aliases beta
    (dict(sN=BASE + (8 << 30)), 1),                         # final state aliases beta
    (dict(ws=None), 3), (dict(ws_bytes=256), 3),
    (dict(sN=BASE + (7 << 30) + 4096), 1),                  # final state inside the workspace
    (dict(B=1 << 16, H=1 << 16), 2),                        # too many segments
])
def test_diag_delta_host_validation_rejects_before_launch(L, over, code):
    assert call_diag_delta(L, **over) == code


class _OnDevice:
    """A CPU tensor that reports itself as a CUDA tensor, so that the
    binding's tensor checks can be exercised on a machine without a GPU."""

    is_cuda = True

    def __init__(self, t):
        self.t = t
        self.dtype, self.shape = t.dtype, t.shape

    def is_contiguous(self):
        return self.t.is_contiguous()

    def dim(self):
        return self.t.dim()

    def numel(self):
        return self.t.numel()


def _fwd_inputs(B=1, T=8, H=2, dk=32, dv=32):
    import torch
    bf = torch.bfloat16
    mk = lambda *s, dt=bf: _OnDevice(torch.zeros(*s, dtype=dt))
    return (mk(B, T, H, dk), mk(B, T, H, dk), mk(B, T, H, dv), mk(B, T, H, dt=torch.float32),
            mk(B, T, H))


@pytest.mark.parametrize("bad", ["o_shape", "o_dtype", "state_shape", "state_dtype", "o_cpu",
                                 "o_missing"])
def test_static_scratch_rejects_bad_outputs_before_the_library(monkeypatch, bad):
    import torch
    q, k, v, g, beta = _fwd_inputs()
    o = _OnDevice(torch.zeros(1, 8, 2, 32, dtype=torch.bfloat16))
    s = _OnDevice(torch.zeros(1, 2, 32, 32, dtype=torch.float32))
    if bad == "o_shape":
        o = _OnDevice(torch.zeros(1, 7, 2, 32, dtype=torch.bfloat16))
    elif bad == "o_dtype":
        o = _OnDevice(torch.zeros(1, 8, 2, 32, dtype=torch.float32))
    elif bad == "state_shape":
        s = _OnDevice(torch.zeros(1, 2, 32, 16, dtype=torch.float32))
    elif bad == "state_dtype":
        s = _OnDevice(torch.zeros(1, 2, 32, 32, dtype=torch.bfloat16))
    elif bad == "o_cpu":
        o = torch.zeros(1, 8, 2, 32, dtype=torch.bfloat16)
    elif bad == "o_missing":
        o = None

    def no_library():
        raise AssertionError("the library was called with malformed tensors")

    monkeypatch.setattr(G, "lib", no_library)
    with pytest.raises((ValueError, TypeError)):
        G.gdn_fwd_static_scratch(q, k, v, g, beta, None, None, o, s)


def test_static_scratch_entry_point_validates_before_enqueueing(L):
    """Host-side rejections of the no-workspace entry point need no device:
    a scratch need above the array's size, and zero sizes."""
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fake = vp(1 << 40)
    args = [fake] * 5 + [vp(None), vp(None), vp((1 << 40) + (1 << 30)), vp(None), vp(None),
                         vp(None)]
    # num_seqs = 0: no scratch size is defined
    st = L.gdn_fwd_static_scratch(*args, i32(1), i32(8), i32(2), i32(32), i32(32), i32(0),
                                  i32(64), ctypes.c_int(1), ctypes.c_uint32(0), i32(0), vp(0))
    assert st == 1
