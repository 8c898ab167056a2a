"""Seeded synthetic inputs shaped like the pages' context stages.

This module holds no arithmetic of the attention method: it only draws random
tensors (torch CPU generator, fp32, then round-to-nearest to bf16) so that the
CUDA library and the fp64 oracle can be fed the very same bytes.

Recipe (one workload per context stage, 8K -> 64K -> 256K -> 1M tokens, from
"Engineering Long-Context Training for Trillion-Parameter MoE Models", sec. 2):
  q ~ N(0,1) / sqrt(dk)             bf16
  k ~ N(0,1), L2-normalised over dk per (token, head) in fp32, then bf16
  v ~ N(0,1)                        bf16
  a ~ N(mean, std)                  fp32 decay logits ([B,T,H], or [B,T,H,dk] for
                                    the per-channel decay)
  dO ~ N(0,1)                       bf16 upstream gradient
  h0 ~ N(0, h0_std) per document    fp32 (absent when h0_std == 0)
  beta = sigmoid(N(0,1))            fp32 [B,T,H] write strengths (gated delta rule
                                    workloads only; drawn after everything above)
Packed documents: n_docs lengths u_i ~ U[lo, hi], rescaled so they sum to T
(floor, remainder added to the last document).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    seed: int
    a_mean: float = 0.0
    a_std: float = 1.0
    b: float = -5.0
    mode: int = 0                  # 0 bounded sigmoid, 1 unbounded -softplus (ablation)
    h0_std: float = 0.0
    n_docs: int = 0                # >0: packed documents (B must be 1)
    doc_lo: int = 0
    doc_hi: int = 0
    fwd_only: bool = False
    o_f32: bool = False            # fp32 o (else bf16)
    ckpt_stride: int = 0           # >0: fp32 state checkpoints every ckpt_stride tokens
    vec: bool = False              # one decay logit per key channel: a [B,T,H,dk]
    delta: bool = False            # gated delta rule: write strengths beta [B,T,H]

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    # forward-only parity case, fp32 output and state
    "pr1": Workload("pr1", B=1, T=256, H=2, dk=64, dv=64, seed=1000, fwd_only=True, o_f32=True),
    # 8K stage, batched
    "c8k": Workload("c8k", B=4, T=8192, H=16, dk=128, dv=128, seed=1001),
    # 64K stage: 8 packed documents with a nonzero per-document initial state
    "varlen64k": Workload("varlen64k", B=1, T=65536, H=32, dk=128, dv=128, seed=1002,
                          h0_std=0.1, n_docs=8, doc_lo=1024, doc_hi=16384),
    # 256K stage, dv = 256, decay pushed toward the bound, per-chunk state checkpoints
    "c256k": Workload("c256k", B=1, T=262144, H=16, dk=128, dv=256, seed=1003, a_std=2.0,
                      ckpt_stride=16),
    # 1M stage
    "c1m": Workload("c1m", B=1, T=1048576, H=8, dk=128, dv=128, seed=1004),
    # 1M stage, unbounded -softplus decay (the ablation)
    "c1m_ablation": Workload("c1m_ablation", B=1, T=1048576, H=8, dk=128, dv=128, seed=1005,
                             a_mean=2.0, a_std=2.0, mode=1),
    # per-channel decay (one logit per key channel) on the 64K stage's packed documents
    "varlen64k_vec": Workload("varlen64k_vec", B=1, T=65536, H=32, dk=128, dv=128, seed=1006,
                              h0_std=0.1, n_docs=8, doc_lo=1024, doc_hi=16384, vec=True),
    # gated delta rule with the bounded decay on the 64K stage's packed documents
    "varlen64k_delta": Workload("varlen64k_delta", B=1, T=65536, H=32, dk=128, dv=128, seed=1007,
                                h0_std=0.1, n_docs=8, doc_lo=1024, doc_hi=16384, delta=True),
}


def doc_lengths(w: Workload, g: torch.Generator) -> list[int]:
    u = torch.empty(w.n_docs, dtype=torch.float64).uniform_(w.doc_lo, w.doc_hi, generator=g)
    lens = [int(math.floor(x)) for x in (u * w.T / u.sum()).tolist()]
    lens[-1] += w.T - sum(lens)
    return lens


def _randn(shape, g, chunk_rows=1 << 18):
    """fp32 N(0,1) drawn in row chunks to bound peak host memory."""
    out = torch.empty(shape, dtype=torch.float32)
    flat = out.view(-1, shape[-1])
    for r in range(0, flat.shape[0], chunk_rows):
        flat[r:r + chunk_rows] = torch.randn(flat[r:r + chunk_rows].shape, generator=g)
    return out


def make_inputs(w: Workload, with_grad: Optional[bool] = None) -> dict:
    """Returns CPU tensors: q,k [B,T,H,dk] bf16, v [B,T,H,dv] bf16, a [B,T,H]
    fp32, dO [B,T,H,dv] bf16 (unless forward-only), h0 [N,H,dk,dv] fp32 or None,
    cu_seqlens int32 [N+1] (packed workloads) or None, beta [B,T,H] fp32
    (gated delta rule workloads) or None."""
    if with_grad is None:
        with_grad = not w.fwd_only
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    cu = None
    if w.n_docs:
        assert B == 1
        lens = doc_lengths(w, g)
        cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
    q = (_randn((B, T, H, dk), g) * (1.0 / math.sqrt(dk))).to(torch.bfloat16)
    k32 = _randn((B, T, H, dk), g)
    k32 = k32 / k32.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    k = k32.to(torch.bfloat16)
    del k32
    v = _randn((B, T, H, dv), g).to(torch.bfloat16)
    a = (_randn((B, T, H, dk) if w.vec else (B, T, H), g) * w.a_std + w.a_mean).contiguous()
    dO = _randn((B, T, H, dv), g).to(torch.bfloat16) if with_grad else None
    n_seq = (cu.numel() - 1) if cu is not None else B
    h0 = (_randn((n_seq, H, dk, dv), g) * w.h0_std) if w.h0_std > 0 else None
    beta = torch.sigmoid(_randn((B, T, H), g)).contiguous() if w.delta else None
    return dict(q=q, k=k, v=v, a=a, dO=dO, h0=h0, cu_seqlens=cu, beta=beta)


def make_inputs_on(w: Workload, device, with_grad: bool = True) -> dict:
    """The same recipe drawn directly on `device` with a device generator
    seeded from the workload (values differ from make_inputs' CPU draws; the
    distributions and shapes are the same).  For timing runs that compare
    nothing with the oracle and would otherwise spend a minute drawing
    billion-element tensors on the host."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    cu = None
    if w.n_docs:
        gc = torch.Generator(device="cpu")
        gc.manual_seed(w.seed)
        lens = doc_lengths(w, gc)
        cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32).to(device)
    rn = lambda shape: torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    q = (rn((B, T, H, dk)) * (1.0 / math.sqrt(dk))).to(torch.bfloat16)
    k32 = rn((B, T, H, dk))
    k = (k32 / k32.norm(dim=-1, keepdim=True).clamp_min(1e-12)).to(torch.bfloat16)
    del k32
    v = rn((B, T, H, dv)).to(torch.bfloat16)
    a = (rn((B, T, H, dk) if w.vec else (B, T, H)) * w.a_std + w.a_mean).contiguous()
    dO = rn((B, T, H, dv)).to(torch.bfloat16) if with_grad else None
    n_seq = (cu.numel() - 1) if cu is not None else B
    h0 = (rn((n_seq, H, dk, dv)) * w.h0_std) if w.h0_std > 0 else None
    beta = torch.sigmoid(rn((B, T, H))).contiguous() if w.delta else None
    return dict(q=q, k=k, v=v, a=a, dO=dO, h0=h0, cu_seqlens=cu, beta=beta)


def small_variant(w: Workload, T: int, H: Optional[int] = None, n_docs: Optional[int] = None,
                  seed_offset: int = 0) -> Workload:
    """Same recipe at a size the oracle finishes in seconds."""
    nd = w.n_docs if n_docs is None else n_docs
    lo, hi = w.doc_lo, w.doc_hi
    if nd:
        lo = max(1, min(lo, T // (2 * nd)))
        hi = max(lo + 1, min(hi, 2 * T // nd))
    return dataclasses.replace(w, name=f"{w.name}_T{T}", T=T, H=H or w.H, n_docs=nd,
                               doc_lo=lo, doc_hi=hi, seed=w.seed + 7919 * (seed_offset + 1))
