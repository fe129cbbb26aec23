"""MSA (MiniMax-style sparse attention) training on GB300: Python binding of libmsa.

The functions below carry the names of the C ABI (include/msa.h) and only
marshal arguments: torch tensors provide device memory and the CUDA stream,
every step of the computation runs in the library's sm_103a kernels.  If the
library has not been built the calls raise; there is no fallback.

    params = make_params(T, num_docs, max_seqlen, hq, hkv, d, dp, top_k)
    msa_proxy_select(params, cu_seqlens, q_p, k_p, sel_idx, sel_score, sel_arg, plse, tie, ws)
    msa_fwd(params, cu_seqlens, q, k, v, sel_idx, o, o_res, lse, mass, ws)
    msa_bwd(params, cu_seqlens, q, k, v, q_p, k_p, o, o_res, lse, mass, dO, sel_idx, sel_score,
            sel_arg, plse, dq, dk, dv, dq_p, dk_p, kl_loss, ws)
"""
from __future__ import annotations

import ctypes

import torch

from ._abi import (EXPORTS, LIB_PATH, MSA_FLAG_REUSE_REGROUP, MSA_FLAG_TEST_STALL_SELECT, MSA_OK,
                   MsaError, MsaParams, STATUS_NAMES, load)

__all__ = [
    "MsaError", "MsaParams", "MSA_FLAG_REUSE_REGROUP", "MSA_FLAG_TEST_STALL_SELECT", "make_params", "msa_select_workspace_size", "msa_fwd_workspace_size",
    "msa_bwd_workspace_size", "msa_proxy_select", "msa_proxy_select_noalloc", "msa_fwd", "msa_bwd", "msa_get_device_status",
    "msa_last_status_word", "msa_launch_count", "msa_set_profile_events", "msa_status_string", "allocate_outputs", "workspace", "EXPORTS", "LIB_PATH", "load",
]


def make_params(total_tokens, num_docs, max_seqlen, hq, hkv, d, dp, top_k, block=128,
                softmax_scale=1.0, proxy_scale=1.0, kl_weight=1.0, flags=0, window=0,
                dilation=1) -> MsaParams:
    """msa_params; window/dilation set the always-kept block pattern (0: none)."""
    return MsaParams(total_tokens=int(total_tokens), num_docs=int(num_docs),
                     max_seqlen=int(max_seqlen), hq=int(hq), hkv=int(hkv), d=int(d), dp=int(dp),
                     block=int(block), top_k=int(top_k), window=int(window),
                     dilation=int(dilation), softmax_scale=float(softmax_scale),
                     proxy_scale=float(proxy_scale), kl_weight=float(kl_weight),
                     flags=int(flags))


def _ptr(t) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmsa must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != MSA_OK:
        raise MsaError(status, where)


def msa_select_workspace_size(params: MsaParams) -> int:
    return int(load().msa_select_workspace_size(ctypes.byref(params)))


def msa_fwd_workspace_size(params: MsaParams) -> int:
    return int(load().msa_fwd_workspace_size(ctypes.byref(params)))


def msa_bwd_workspace_size(params: MsaParams) -> int:
    return int(load().msa_bwd_workspace_size(ctypes.byref(params)))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A caller-owned workspace buffer (uint8) of at least `nbytes` bytes."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def msa_proxy_select(params, cu_seqlens, q_p, k_p, sel_idx, sel_score, sel_arg, plse, tie, ws,
                     stream=None) -> None:
    _check(load().msa_proxy_select(ctypes.byref(params), _ptr(cu_seqlens), _ptr(q_p), _ptr(k_p),
                                   _ptr(sel_idx), _ptr(sel_score), _ptr(sel_arg), _ptr(plse),
                                   _ptr(tie), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)), "msa_proxy_select")


def msa_proxy_select_noalloc(params, cu_seqlens, q_p, k_p, sel_idx, sel_score, sel_arg, plse, tie,
                             stream=None) -> None:
    """msa_proxy_select for callers that cannot allocate: no workspace argument,
    the scratch is a static device array inside the library (see include/msa.h)."""
    _check(load().msa_proxy_select_noalloc(ctypes.byref(params), _ptr(cu_seqlens), _ptr(q_p),
                                           _ptr(k_p), _ptr(sel_idx), _ptr(sel_score),
                                           _ptr(sel_arg), _ptr(plse), _ptr(tie), _stream(stream)),
           "msa_proxy_select_noalloc")


def msa_fwd(params, cu_seqlens, q, k, v, sel_idx, o, o_res, lse, mass, ws, stream=None) -> None:
    _check(load().msa_fwd(ctypes.byref(params), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v),
                          _ptr(sel_idx), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(mass), _ptr(ws),
                          ws.numel() * ws.element_size(), _stream(stream)), "msa_fwd")


def msa_bwd(params, cu_seqlens, q, k, v, q_p, k_p, o, o_res, lse, mass, dO, sel_idx, sel_score,
            sel_arg, plse, dq, dk, dv, dq_p, dk_p, kl_loss, ws, stream=None) -> None:
    _check(load().msa_bwd(ctypes.byref(params), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v),
                          _ptr(q_p), _ptr(k_p), _ptr(o), _ptr(o_res), _ptr(lse), _ptr(mass),
                          _ptr(dO),
                          _ptr(sel_idx), _ptr(sel_score), _ptr(sel_arg), _ptr(plse), _ptr(dq),
                          _ptr(dk), _ptr(dv), _ptr(dq_p), _ptr(dk_p), _ptr(kl_loss), _ptr(ws),
                          ws.numel() * ws.element_size(), _stream(stream)), "msa_bwd")


def msa_get_device_status(stream=None) -> int:
    return int(load().msa_get_device_status(_stream(stream)))


def msa_last_status_word() -> int:
    """Full status word (code | where a wait ran out) seen by the last status read."""
    return int(load().msa_last_status_word())


def msa_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().msa_launch_count())


def msa_set_profile_events(which: int, start=None, stop=None) -> None:
    """Record torch.cuda.Event `start`/`stop` around kernel `which` (1 select,
    2 forward block kernel, 3 backward block kernel); None clears."""
    h = (lambda e: ctypes.c_void_p(e.cuda_event) if e is not None else ctypes.c_void_p(0))
    _check(load().msa_set_profile_events(int(which), h(start), h(stop)), "msa_set_profile_events")


def msa_status_string(status: int) -> str:
    return load().msa_status_string(int(status)).decode()


def allocate_outputs(params: MsaParams, device="cuda") -> dict:
    """Output tensors of one step (select + fwd + bwd) for `params`."""
    T, hq, hkv, d, dp, K = (params.total_tokens, params.hq, params.hkv, params.d, params.dp,
                            params.top_k)
    f32, dev = torch.float32, device
    return dict(
        sel_idx=torch.empty(T, hkv, K, dtype=torch.int32, device=dev),
        sel_score=torch.empty(T, hkv, K, dtype=f32, device=dev),
        sel_arg=torch.empty(T, hkv, K, dtype=torch.uint8, device=dev),
        plse=torch.empty(T, hkv, dtype=f32, device=dev),
        tie=torch.empty(T, hkv, dtype=torch.uint8, device=dev),
        o=torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev),
        o_res=torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev),
        lse=torch.empty(T, hq, dtype=f32, device=dev),
        mass=torch.empty(T, hkv, K, dtype=f32, device=dev),
        dq=torch.empty(T, hq, d, dtype=f32, device=dev),
        dk=torch.empty(T, hkv, d, dtype=f32, device=dev),
        dv=torch.empty(T, hkv, d, dtype=f32, device=dev),
        dq_p=torch.empty(T, hkv, dp, dtype=f32, device=dev),
        dk_p=torch.empty(T, hkv, dp, dtype=f32, device=dev),
        kl_loss=torch.zeros(1, dtype=torch.float64, device=dev),
    )


# autograd front end (imported last: it builds on the calls above)
from .function import MSAFunction, last_kl_loss, msa_attention  # noqa: E402

__all__ += ["MSAFunction", "msa_attention", "last_kl_loss"]
