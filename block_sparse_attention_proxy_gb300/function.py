"""Autograd front end: MSA attention as a drop-in torch function.

    o = msa_attention(q, k, v, q_p, k_p, cu_seqlens, top_k)

runs the proxy selection and the block-sparse forward through the C ABI; in
the backward pass it runs msa_bwd, which returns dq, dk, dv and, with weight
`kl_weight`, the gradient of the proxy's KL loss into q_p and k_p (the
proxy's training signal; the selection itself is discrete).  The KL loss
value is computed by that backward and is returned by `last_kl_loss()` (a
device fp64 scalar).  This module only moves tensors in and out of the
library; every step runs in the library's kernels.

Each call keeps its own saved tensors (selection, o, o_res, lse, mass), so
several layers may run their forwards before their backwards.  Calls of one
shape share one workspace; the backward rebuilds the block lists, since
another call may have used the workspace in between.

Layouts (packed varlen, token-major): q [T, Hq, d], k/v [T, Hkv, d],
q_p/k_p [T, Hkv, dp], all bf16; cu_seqlens int32 [num_docs + 1] on the device.
"""
from __future__ import annotations

import torch

from . import (allocate_outputs, msa_bwd, msa_fwd, msa_proxy_select, workspace)
from .step import params_for, workspace_bytes

_ws: dict = {}
_last_kl: list = [None]


def _workspace_for(params, device) -> torch.Tensor:
    need = workspace_bytes(params)
    key = str(device)
    ws = _ws.get(key)
    if ws is None or ws.numel() < need:
        _ws[key] = ws = workspace(need, device)
    return ws


class MSAFunction(torch.autograd.Function):
    """o = MSA(q, k, v; q_p, k_p); backward adds kl_weight * d KL / d(q_p, k_p)."""

    @staticmethod
    def forward(ctx, q, k, v, q_p, k_p, cu_seqlens, top_k: int, softmax_scale: float,
                proxy_scale: float, kl_weight: float, window: int, dilation: int):
        for t in (q, k, v, q_p, k_p):
            if t.dtype != torch.bfloat16 or not t.is_cuda:
                raise TypeError("q, k, v, q_p, k_p must be bf16 CUDA tensors")
        hq, d = q.shape[1], q.shape[2]
        hkv, dp = q_p.shape[1], q_p.shape[2]
        cu = cu_seqlens.to(torch.int32).contiguous()
        prm = params_for([int(x) for x in cu.tolist()], hq, hkv, d, dp, top_k,
                         softmax_scale=softmax_scale, proxy_scale=proxy_scale,
                         kl_weight=kl_weight, window=window, dilation=dilation)
        ws = _workspace_for(prm, q.device)
        out = allocate_outputs(prm, q.device)
        q, k, v, q_p, k_p = (t.contiguous() for t in (q, k, v, q_p, k_p))
        stream = torch.cuda.current_stream(q.device)
        msa_proxy_select(prm, cu, q_p, k_p, out["sel_idx"], out["sel_score"], out["sel_arg"],
                         out["plse"], out["tie"], ws, stream)
        msa_fwd(prm, cu, q, k, v, out["sel_idx"], out["o"], out["o_res"], out["lse"],
                out["mass"], ws, stream)
        ctx.prm, ctx.out, ctx.stream = prm, out, stream
        ctx.save_for_backward(q, k, v, q_p, k_p, cu)
        ctx.mark_non_differentiable(cu_seqlens)
        return out["o"]

    @staticmethod
    def backward(ctx, d_o):
        q, k, v, q_p, k_p, cu = ctx.saved_tensors
        prm, o = ctx.prm, ctx.out
        ws = _workspace_for(prm, q.device)
        d_o = d_o.to(torch.bfloat16).contiguous()
        msa_bwd(prm, cu, q, k, v, q_p, k_p, o["o"], o["o_res"], o["lse"], o["mass"], d_o,
                o["sel_idx"], o["sel_score"], o["sel_arg"], o["plse"], o["dq"], o["dk"], o["dv"],
                o["dq_p"], o["dk_p"], o["kl_loss"], ws, ctx.stream)
        _last_kl[0] = o["kl_loss"]
        return (o["dq"], o["dk"], o["dv"], o["dq_p"], o["dk_p"], None, None, None, None, None,
                None, None)


def msa_attention(q, k, v, q_p, k_p, cu_seqlens, top_k: int, softmax_scale: float = 1.0,
                  proxy_scale: float = 1.0, kl_weight: float = 1.0, window: int = 0,
                  dilation: int = 1) -> torch.Tensor:
    """Block-sparse MSA attention over a packed varlen batch (see module docstring).
    window/dilation: blocks j - dilation * u (u = 1..window) are always kept,
    inside the top_k slots (window <= top_k - 1; 0 keeps none)."""
    return MSAFunction.apply(q, k, v, q_p, k_p, cu_seqlens, int(top_k), float(softmax_scale),
                             float(proxy_scale), float(kl_weight), int(window), int(dilation))


def last_kl_loss() -> torch.Tensor | None:
    """The proxy KL loss computed by the most recent backward (device fp64 scalar)."""
    return _last_kl[0]
