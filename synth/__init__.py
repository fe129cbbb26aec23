"""Seeded synthetic inputs for MSA (MiniMax-style sparse attention) training steps.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle may take their
inputs from it.

Workloads (shapes, value distributions, structure):

  tiny     1 sequence of 1024 tokens, Hq=4, Hkv=1, d=64, dp=32, top-k 4, iid N(0,1), seed 0
  varlen   32768 tokens packed as 8 documents, lengths drawn U[1024, 8192] and
           rescaled to sum 32768, Hq=16, Hkv=4, d=128, dp=64, top-k 8, iid N(0,1), seed 1
  128k     1 sequence of 131072 tokens, Hq=32, Hkv=8, d=128, dp=64, top-k 16,
           k and k_p carry a shared rank-8 component, seed 2
  512k     as 128k with 524288 tokens, seed 3
  1m       as 128k with 1048576 tokens, seed 4
  8k       as 128k with 8192 tokens, seed 5 (a profiling-size case of the same kernels:
           its inputs still exceed L2, its workspace stays near 1.5 GB)

Recipe (all draws fp32 from one torch.Generator seeded with the workload
seed, in this order, then rounded to bf16):
  q   ~ N(0,1) / sqrt(d)      [T, Hq, d]     (pre-scaled, so softmax scale = 1)
  k   ~ N(0,1)                [T, Hkv, d]
  v   ~ N(0,1)                [T, Hkv, d]
  q_p ~ N(0,1) / sqrt(dp)     [T, Hkv, dp]   (pre-scaled, so proxy scale = 1)
  k_p ~ N(0,1)                [T, Hkv, dp]
  dO  ~ N(0,1)                [T, Hq, d]
  structured workloads only, then:
  A   ~ N(0,1) [T, Hkv, 8],  U_k ~ N(0,1) [Hkv, 8, d],  U_p ~ N(0,1) [Hkv, 8, dp]
  k   += 0.5 * A U_k,  k_p += 0.5 * A U_p   (A shared by k and k_p, per group)
Document lengths (varlen) come first, from a separate CPU generator with the
same seed, so they do not depend on the device the tensors are drawn on.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

BLOCK = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    doc_lengths: tuple
    hq: int
    hkv: int
    d: int
    dp: int
    top_k: int
    seed: int
    structured: bool
    block: int = BLOCK

    @property
    def total_tokens(self) -> int:
        return int(sum(self.doc_lengths))

    @property
    def num_docs(self) -> int:
        return len(self.doc_lengths)

    @property
    def max_seqlen(self) -> int:
        return int(max(self.doc_lengths)) if self.doc_lengths else 0


def varlen_lengths(total: int, ndoc: int, lo: float, hi: float, seed: int) -> List[int]:
    """Draw ndoc lengths uniform in [lo, hi], rescale so they sum to `total`
    (floor for all but the last document, which takes the remainder)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.rand(ndoc, generator=g, dtype=torch.float64) * (hi - lo) + lo
    scale = total / float(u.sum())
    lens = [int(math.floor(float(x) * scale)) for x in u[:-1]]
    lens.append(total - sum(lens))
    return lens


def workload(name: str) -> Workload:
    if name == "tiny":
        return Workload("tiny", (1024,), 4, 1, 64, 32, 4, 0, False)
    if name == "varlen":
        return Workload("varlen", tuple(varlen_lengths(32768, 8, 1024.0, 8192.0, 1)), 16, 4, 128,
                        64, 8, 1, False)
    if name == "128k":
        return Workload("128k", (131072,), 32, 8, 128, 64, 16, 2, True)
    if name == "512k":
        return Workload("512k", (524288,), 32, 8, 128, 64, 16, 3, True)
    if name == "1m":
        return Workload("1m", (1048576,), 32, 8, 128, 64, 16, 4, True)
    if name == "8k":
        return Workload("8k", (8192,), 32, 8, 128, 64, 16, 5, True)
    raise KeyError(name)


WORKLOADS = ("tiny", "varlen", "128k", "512k", "1m", "8k")


def custom(doc_lengths, hq, hkv, d, dp, top_k, seed, structured=False, block=BLOCK) -> Workload:
    return Workload("custom", tuple(int(x) for x in doc_lengths), hq, hkv, d, dp, top_k, seed,
                    structured, block)


def cu_seqlens_of(w: Workload) -> torch.Tensor:
    cu = [0]
    for L in w.doc_lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(w: Workload, device="cpu", dtype=torch.bfloat16, rank: int = 8,
                structure_scale: float = 0.5) -> dict:
    """Draw the workload's tensors on `device` (see the module docstring)."""
    T = w.total_tokens
    g = torch.Generator(device=device).manual_seed(w.seed)

    def draw(*shape, scale=1.0):
        x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        return x

    q = draw(T, w.hq, w.d, scale=1.0 / math.sqrt(w.d)).to(dtype)
    k = draw(T, w.hkv, w.d)
    v = draw(T, w.hkv, w.d).to(dtype)
    q_p = draw(T, w.hkv, w.dp, scale=1.0 / math.sqrt(w.dp)).to(dtype)
    k_p = draw(T, w.hkv, w.dp)
    dO = draw(T, w.hq, w.d).to(dtype)
    if w.structured:
        A = draw(T, w.hkv, rank)
        Uk = draw(w.hkv, rank, w.d)
        Up = draw(w.hkv, rank, w.dp)
        k.add_(torch.einsum("tgr,grd->tgd", A, Uk), alpha=structure_scale)
        k_p.add_(torch.einsum("tgr,grd->tgd", A, Up), alpha=structure_scale)
        del A, Uk, Up
    k = k.to(dtype)
    k_p = k_p.to(dtype)
    return dict(q=q, k=k, v=v, q_p=q_p, k_p=k_p, dO=dO,
                cu_seqlens=cu_seqlens_of(w).to(device))


def sample_rows(T: int, n: int, seed: int) -> torch.Tensor:
    """Rows 0 and T-1 plus n-2 distinct rows drawn with a generator seeded by `seed`."""
    if n >= T:
        return torch.arange(T)
    g = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(T - 2, generator=g)[: n - 2] + 1
    rows = torch.cat([torch.tensor([0, T - 1]), perm])
    return torch.sort(rows).values
