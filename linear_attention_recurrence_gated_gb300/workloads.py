"""Seeded synthetic inputs for the gated delta rule forward pass.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic.  Both the CUDA path and the oracle are fed from it.

Recipe (one ``numpy.random.default_rng(seed)`` stream per workload, drawn in
this order, everything as fp64 standard normals first):

1. varlen only: sequence lengths ``rng.integers(lo, hi + 1, num_seqs)``;
2. q, then k: N(0, 1), each (token, head) row divided by its L2 norm in fp64;
3. v: N(0, 1);
4. gate normal z_g: g = -softplus(z_g) * gate_scale, stored as fp32
   (softplus(z) = log1p(exp(z)), evaluated stably);
5. beta normal z_b: beta = sigmoid(z_b), stored in the input dtype;
6. initial state (when requested): N(0, 0.02^2), fp32, shape [N, H, dk, dv].

Values are cast to the storage dtype with round-to-nearest-even (torch's
``.to(torch.bfloat16)``).  The shapes stand in for the GDN layer shapes on
the HyMo pages ("Model Architecture Walkthrough" section 5.5: B=4, T=4096,
H=40, S=D=32), scaled to the five named workloads below; no dataset is used.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    dk: int
    dv: int
    dtype: str
    B: int = 1
    T: int = 0
    num_seqs: int = 0            # > 0 selects packed variable-length sequences
    len_range: tuple = (0, 0)    # inclusive length range for varlen draws
    gate_scale: float = 1.0
    init_state: bool = False
    seed: int = 0
    notes: str = field(default="", compare=False)

    @property
    def varlen(self) -> bool:
        return self.num_seqs > 0


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, T=256, H=2, dk=32, dv=32, dtype="fp32",
                          gate_scale=0.1, init_state=False,
                          notes="latency-bound; parity focus"),
    "hymo_bf16": Workload("hymo_bf16", B=8, T=4096, H=16, dk=64, dv=64, dtype="bf16",
                          gate_scale=1.0, init_state=False,
                          notes="HyMo-shaped GDN layer; the benchmark workload"),
    "wide_bf16": Workload("wide_bf16", B=4, T=8192, H=16, dk=128, dv=128, dtype="bf16",
                          gate_scale=1.0, init_state=True),
    "long_bf16": Workload("long_bf16", B=1, T=65536, H=16, dk=128, dv=128, dtype="bf16",
                          gate_scale=0.01, init_state=False,
                          notes="slow gates stress long-range state carry"),
    "varlen_bf16": Workload("varlen_bf16", num_seqs=32, len_range=(128, 8192), H=8,
                            dk=128, dv=256, dtype="bf16", gate_scale=1.0, init_state=True),
}


# One recurrent step per sequence (the decode entry point): B sequences of one
# token, with a running state.  1024 HyMo-shaped heads-by-sequences give a
# 256 MB state, larger than the 129 MB L2, so a timed step streams it from HBM.
DECODE_WORKLOADS = {
    "decode_hymo_bf16": Workload("decode_hymo_bf16", B=1024, T=1, H=16, dk=64, dv=64,
                                 dtype="bf16", gate_scale=1.0, init_state=True,
                                 notes="1024 sequences x 16 heads, one step each"),
}


def generate_decode(w: Workload):
    """Inputs of one decode step: the draws of ``generate`` for ``w`` (which must
    have T == 1) with the token axis removed: q, k ``[N, H, dk]``, v ``[N, H, dv]``,
    g, beta ``[N, H]``, state ``[N, H, dk, dv]`` fp32 or None."""
    if w.T != 1 or w.varlen:
        raise ValueError("a decode workload has B sequences of exactly one token")
    d = generate(w)
    return {"q": d["q"][:, 0].contiguous(), "k": d["k"][:, 0].contiguous(),
            "v": d["v"][:, 0].contiguous(), "g": d["g"][:, 0].contiguous(),
            "beta": d["beta"][:, 0].contiguous(), "state": d["initial_state"], "N": w.B}


def custom(name="custom", **kw) -> Workload:
    """A workload with explicit fields (edge-case tests)."""
    return Workload(name=name, **kw)


def with_seed(w: Workload, seed: int) -> Workload:
    return replace(w, seed=seed)


def _l2_rows(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def generate(w: Workload, lengths=None):
    """Draw the inputs of workload ``w`` on the host.

    Returns a dict of CPU torch tensors: q, k ``[B, T, H, dk]``; v ``[B, T, H, dv]``
    (storage dtype); g ``[B, T, H]`` fp32; beta ``[B, T, H]`` (storage dtype);
    initial_state ``[N, H, dk, dv]`` fp32 or None; cu_seqlens int32 ``[N+1]`` or
    None; plus ``N`` and ``tokens``.  ``lengths`` overrides the varlen draw (the
    draw still happens, so the stream order is unchanged).
    """
    rng = np.random.default_rng(w.seed)
    dt = _DTYPES[w.dtype]
    cu = None
    if w.varlen:
        drawn = rng.integers(w.len_range[0], w.len_range[1] + 1, w.num_seqs)
        lens = np.asarray(drawn if lengths is None else lengths, dtype=np.int64)
        cu_np = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        B, T, N = 1, int(cu_np[-1]), len(lens)
        cu = torch.from_numpy(cu_np.astype(np.int32))
    else:
        B, T, N = w.B, w.T, w.B
    H, dk, dv = w.H, w.dk, w.dv

    def draw(shape):
        return rng.standard_normal(shape)

    q = torch.from_numpy(_l2_rows(draw((B, T, H, dk)))).to(dt)
    k = torch.from_numpy(_l2_rows(draw((B, T, H, dk)))).to(dt)
    v = torch.from_numpy(draw((B, T, H, dv))).to(dt)
    g = torch.from_numpy(-_softplus(draw((B, T, H))) * w.gate_scale).to(torch.float32)
    beta = torch.from_numpy(_sigmoid(draw((B, T, H)))).to(dt)
    s0 = None
    if w.init_state:
        s0 = torch.from_numpy(0.02 * draw((N, H, dk, dv))).to(torch.float32)
    return {"q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(),
            "g": g.contiguous(), "beta": beta.contiguous(), "initial_state": s0,
            "cu_seqlens": cu, "N": N, "tokens": B * T}


def generate_block_extras(inputs, H: int, seed: int, dtype: str = "bf16"):
    """Extra inputs of the fused block parts of a forward call, drawn from their
    own stream (seed) so the base draw is unchanged: ``beta_logits`` N(0, 1) in
    the storage dtype (the kernel applies the sigmoid), ``D_skip`` ``[H]``
    N(1, 0.5^2) fp32 (the pages initialise D to 1), ``out_gate`` ``[B, T, H]``
    U(0, 1) fp32 (a mean of sigmoid outputs on the pages), and raw q/k of
    random lengths for the in-kernel normalisation: ``q_raw``/``k_raw`` the
    base q/k rows each scaled by U(0.5, 5)."""
    rng = np.random.default_rng(seed)
    dt = _DTYPES[dtype]
    B, T = inputs["q"].shape[:2]
    z = torch.from_numpy(rng.standard_normal((B, T, H))).to(dt)
    d_skip = torch.from_numpy(1.0 + 0.5 * rng.standard_normal(H)).to(torch.float32)
    gate = torch.from_numpy(rng.uniform(0.0, 1.0, (B, T, H))).to(torch.float32)
    sq = torch.from_numpy(rng.uniform(0.5, 5.0, (B, T, H, 1)))
    sk = torch.from_numpy(rng.uniform(0.5, 5.0, (B, T, H, 1)))
    q_raw = (inputs["q"].double() * sq).to(dt)
    k_raw = (inputs["k"].double() * sk).to(dt)
    return {"beta_logits": z.contiguous(), "D_skip": d_skip.contiguous(),
            "out_gate": gate.contiguous(), "q_raw": q_raw.contiguous(), "k_raw": k_raw.contiguous()}


def head_tokens(w: Workload, inputs=None) -> int:
    if inputs is not None:
        return inputs["tokens"] * w.H
    if w.varlen:
        raise ValueError("varlen head-token count needs the drawn inputs")
    return w.B * w.T * w.H


# ---------------------------------------------------------------------------
# The pages' own recurrence (diagonal decay exp(g_t A), write key b, read key c)
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class DiagWorkload:
    """Inputs of ``gdn_diag_fwd``.  ``a_log`` selects the decay rates:
    "pages": A_log[h, s] = log(h + 1) for every s, the initialisation the pages
    give ("Model Architecture Walkthrough", section 5.3.2: A = -1 ... -H);
    "uniform": A_log[h, s] ~ U(-2, 2) independently (a different rate per row);
    "slow": A_log[h, s] ~ U(-6, -3) (per-token factors near 1: long memory).
    ``delta`` selects the inputs of ``gdn_diag_delta_fwd`` (the same decay
    combined with the delta rule): unit write keys and a write strength beta."""
    name: str
    B: int
    T: int
    H: int
    S: int = 32
    D: int = 32
    dtype: str = "bf16"
    a_log: str = "pages"
    init_state: bool = False
    seed: int = 0
    delta: bool = False
    notes: str = field(default="", compare=False)


DIAG_WORKLOADS = {
    "hymo_diag_bf16": DiagWorkload("hymo_diag_bf16", B=4, T=4096, H=40, dtype="bf16",
                                   a_log="pages",
                                   notes="the pages' production GDN layer (B=4, T=4096, "
                                         "H=40, S=D=32); the diagonal-decay benchmark"),
    "diag_small_fp32": DiagWorkload("diag_small_fp32", B=2, T=300, H=3, dtype="fp32",
                                    a_log="uniform", init_state=True,
                                    notes="parity case: several CTAs and a ragged tail"),
    "hymo_diag_delta_bf16": DiagWorkload("hymo_diag_delta_bf16", B=4, T=4096, H=40,
                                         dtype="bf16", a_log="pages", delta=True,
                                         notes="the pages' production shape with the delta "
                                               "rule's erase added (diagonal decay + delta rule)"),
}


def generate_diag(w: DiagWorkload):
    """Draw the inputs of ``w`` on the host, in this order from one
    ``default_rng(seed)`` stream: v ~ N(0, 1) ``[B, T, H, D]``; b, c ~ N(0, 1/S)
    ``[B, T, H, S]``; g = sigmoid(z), z ~ N(0, 1) ``[B, T, H]`` fp32 (the pages'
    g is a sigmoid output); A_log ``[H, S]`` fp32 per ``w.a_log``; initial
    state ~ N(0, 0.1^2) ``[B, H, S, D]`` fp32 when ``w.init_state``.  v, b, c
    are cast to the storage dtype (round to nearest even).  With ``w.delta``
    each row b_t is divided by its L2 norm in fp64 before the cast (the delta
    rule's erase is a projection for unit keys) and, drawn last, beta =
    sigmoid(z), z ~ N(0, 1) ``[B, T, H]`` in the storage dtype."""
    rng = np.random.default_rng(w.seed)
    dt = _DTYPES[w.dtype]
    B, T, H, S, D = w.B, w.T, w.H, w.S, w.D
    v = torch.from_numpy(rng.standard_normal((B, T, H, D))).to(dt)
    b64 = rng.standard_normal((B, T, H, S))
    b64 = b64 / np.linalg.norm(b64, axis=-1, keepdims=True) if w.delta else b64 / np.sqrt(S)
    b = torch.from_numpy(b64).to(dt)
    c = torch.from_numpy(rng.standard_normal((B, T, H, S)) / np.sqrt(S)).to(dt)
    g = torch.from_numpy(_sigmoid(rng.standard_normal((B, T, H)))).to(torch.float32)
    if w.a_log == "pages":
        a = np.repeat(np.log(np.arange(1, H + 1, dtype=np.float64))[:, None], S, axis=1)
    elif w.a_log == "uniform":
        a = rng.uniform(-2.0, 2.0, (H, S))
    elif w.a_log == "slow":
        a = rng.uniform(-6.0, -3.0, (H, S))
    else:
        raise ValueError(f"unknown a_log recipe {w.a_log!r}")
    A_log = torch.from_numpy(a).to(torch.float32)
    h0 = None
    if w.init_state:
        h0 = torch.from_numpy(0.1 * rng.standard_normal((B, H, S, D))).to(torch.float32)
    out = {"v": v.contiguous(), "b": b.contiguous(), "c": c.contiguous(),
           "g": g.contiguous(), "A_log": A_log.contiguous(), "initial_state": h0}
    if w.delta:
        out["beta"] = torch.from_numpy(_sigmoid(rng.standard_normal((B, T, H)))).to(dt).contiguous()
    return out


# ---------------------------------------------------------------------------
# The GDN block prologue (causal depthwise conv1d + SiLU)
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class ConvWorkload:
    name: str
    B: int
    T: int
    C: int
    K: int = 4
    dtype: str = "bf16"
    seed: int = 0
    notes: str = field(default="", compare=False)


CONV_WORKLOADS = {
    "conv_hymo_bf16": ConvWorkload("conv_hymo_bf16", B=4, T=4096, C=1280, K=4, dtype="bf16",
                                   notes="the pages' prologue: d_inner 1280, d_conv 4"),
}


def generate_conv(w: ConvWorkload):
    """x ~ N(0, 1) ``[B, T, C]`` in the storage dtype, then the conv weights
    w ~ N(0, 1/K) ``[C, K]`` fp32 (PyTorch's default Conv1d scale is of this
    order), from one ``default_rng(seed)`` stream in that order."""
    rng = np.random.default_rng(w.seed)
    x = torch.from_numpy(rng.standard_normal((w.B, w.T, w.C))).to(_DTYPES[w.dtype])
    wt = torch.from_numpy(rng.standard_normal((w.C, w.K)) / np.sqrt(w.K)).to(torch.float32)
    return {"x": x.contiguous(), "w": wt.contiguous()}
