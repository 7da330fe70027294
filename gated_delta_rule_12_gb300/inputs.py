"""Seeded synthetic inputs for the gated delta rule workloads.

This module holds no arithmetic of the method itself: it only draws random
tensors (on the CPU, with ``torch.Generator``) in the shapes, value ranges and
structure of the workloads below.  Both the CUDA path and the fp64 oracle are
fed from here.

Recipe (same for every workload unless noted):
  * draw order: [varlen lengths], q, k, v, z, z', [initial state];
  * q, k, v ~ N(0, 1); q and k are handed to the operator raw and the operator
    L2-normalises them per token-head (``use_qk_l2norm=1``); the operator
    scales q by ``1/sqrt(d_k)``;
  * log-decay g = log(alpha) = -c * softplus(z), z ~ N(0, 1), with c = 0.1
    (c = 1.0 for the large heavy-decay prefill);
  * write strength beta = sigmoid(z'), z' ~ N(0, 1);
  * initial states, where used, ~ 0.02 * N(0, 1), fp32;
  * bf16 workloads round q, k, v to bf16 once here; gates and states stay fp32;
  * varlen: 8 lengths ~ U[512, 8192], rescaled to sum to the token total,
    rounded, the last one adjusted so the sum is exact; int32 cu_seqlens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" | "varlen" | "decode"
    H: int
    dk: int
    dv: int
    dtype: str                # "f32" | "bf16"
    seed: int
    B: int = 1
    L: int = 0                # tokens per sequence (prefill) / total tokens (varlen)
    num_seqs: int = 0         # varlen sequences / decode batch N
    steps: int = 0            # decode steps
    decay: float = 0.1        # g = -decay * softplus(z)
    init_state: bool = False
    chunk_size: int = 64
    notes: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dk)

    @property
    def tokens(self) -> int:
        if self.kind == "decode":
            return self.num_seqs * self.steps
        return self.B * self.L


WORKLOADS = {
    w.name: w for w in [
        Workload("prefill_b1_h2_l256_d64_f32", "prefill", H=2, dk=64, dv=64, dtype="f32", seed=0,
                 B=1, L=256, notes="small fp32 case the oracle finishes instantly"),
        Workload("prefill_b4_h16_l2048_d128_bf16", "prefill", H=16, dk=128, dv=128, dtype="bf16",
                 seed=1, B=4, L=2048, notes="headline chunked-forward workload"),
        Workload("varlen_t32768_h16_d128_bf16", "varlen", H=16, dk=128, dv=128, dtype="bf16", seed=2,
                 L=32768, num_seqs=8, init_state=True,
                 notes="packed prefill, 8 sequences, per-sequence initial state"),
        Workload("decode_n256_h16_d128_bf16", "decode", H=16, dk=128, dv=128, dtype="bf16", seed=3,
                 num_seqs=256, steps=64, init_state=True,
                 notes="64 successive single-token steps on a resident fp32 state"),
        Workload("prefill_b8_h32_l8192_dk128_dv256_bf16", "prefill", H=32, dk=128, dv=256,
                 dtype="bf16", seed=4, B=8, L=8192, decay=1.0,
                 notes="large prefill with heavy decay"),
    ]
}


def varlen_lengths(total: int, n: int, gen: torch.Generator, lo: int = 512, hi: int = 8192):
    raw = torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64).tolist()
    s = sum(raw)
    lens = [max(1, int(round(x * total / s))) for x in raw[:-1]]
    lens.append(total - sum(lens))
    if lens[-1] < 1:
        raise ValueError("varlen rescale produced an empty last sequence")
    return lens


def cu_from_lengths(lens):
    cu = [0]
    for x in lens:
        cu.append(cu[-1] + int(x))
    return torch.tensor(cu, dtype=torch.int32)


def _round(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def draw_gates(shape, decay, gen, beta_max=1.0):
    """g = -decay * softplus(z), beta = beta_max * sigmoid(z').  beta_max = 2 gives the
    negative-eigenvalue range beta in (0, 2)."""
    z = torch.randn(shape, generator=gen, dtype=torch.float32)
    zb = torch.randn(shape, generator=gen, dtype=torch.float32)
    g = -decay * torch.nn.functional.softplus(z)
    beta = beta_max * torch.sigmoid(zb)
    return g.contiguous(), beta.contiguous()


def make_prefill(B, L, H, dk, dv, dtype="bf16", seed=0, decay=0.1, init_state=False,
                 num_seqs=0, lengths=None, beta_max=1.0):
    """Inputs of one chunked-forward call.

    Returns a dict with q, k [B,T,H,dk], v [B,T,H,dv], g, beta [B,T,H] (fp32),
    init_state [N,H,dv,dk] fp32 or None, cu_seqlens int32 [N+1] or None.
    With ``num_seqs`` > 0 the call is packed varlen (B must be 1, L total).
    """
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if num_seqs:
        if B != 1:
            raise ValueError("varlen inputs are packed along T with B == 1")
        lens = list(lengths) if lengths is not None else varlen_lengths(L, num_seqs, gen)
        cu = cu_from_lengths(lens)
        if int(cu[-1]) != L:
            raise ValueError("lengths must sum to L")
    q = torch.randn((B, L, H, dk), generator=gen, dtype=torch.float32)
    k = torch.randn((B, L, H, dk), generator=gen, dtype=torch.float32)
    v = torch.randn((B, L, H, dv), generator=gen, dtype=torch.float32)
    g, beta = draw_gates((B, L, H), decay, gen, beta_max)
    N = num_seqs if num_seqs else B
    s0 = (0.02 * torch.randn((N, H, dv, dk), generator=gen, dtype=torch.float32)) if init_state else None
    return dict(q=_round(q, dtype), k=_round(k, dtype), v=_round(v, dtype), g=g, beta=beta,
                init_state=s0, cu_seqlens=cu)


def make_decode(N, H, dk, dv, steps, dtype="bf16", seed=0, decay=0.1, beta_max=1.0):
    """Inputs of ``steps`` successive decode calls.

    Returns q, k [steps,N,H,dk], v [steps,N,H,dv], g, beta [steps,N,H],
    state0 [N,H,dv,dk] fp32.
    """
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((steps, N, H, dk), generator=gen, dtype=torch.float32)
    k = torch.randn((steps, N, H, dk), generator=gen, dtype=torch.float32)
    v = torch.randn((steps, N, H, dv), generator=gen, dtype=torch.float32)
    g, beta = draw_gates((steps, N, H), decay, gen, beta_max)
    s0 = 0.02 * torch.randn((N, H, dv, dk), generator=gen, dtype=torch.float32)
    return dict(q=_round(q, dtype), k=_round(k, dtype), v=_round(v, dtype), g=g, beta=beta, state0=s0)


def make(w: Workload):
    if w.kind == "decode":
        return make_decode(w.num_seqs, w.H, w.dk, w.dv, w.steps, w.dtype, w.seed, w.decay)
    return make_prefill(w.B, w.L, w.H, w.dk, w.dv, w.dtype, w.seed, w.decay, w.init_state,
                        num_seqs=w.num_seqs if w.kind == "varlen" else 0)
