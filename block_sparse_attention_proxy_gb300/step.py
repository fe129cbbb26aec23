"""One MSA training step through the C ABI: proxy select -> forward -> backward.

The three calls run back to back on one stream and share one caller-owned
workspace (the largest of the three sizes): the forward's slot partials are
dead once its merge has run, so the backward reuses the same bytes.  The
selection builds the block lists (queries per KV block) at the front of the
workspace; the forward and backward reuse them (MSA_FLAG_REUSE_REGROUP) when
nothing has touched them since.
"""
from __future__ import annotations

import torch

from . import (MSA_FLAG_REUSE_REGROUP, MsaParams, allocate_outputs, make_params, msa_bwd,
               msa_bwd_workspace_size, msa_fwd, msa_fwd_workspace_size, msa_proxy_select,
               msa_select_workspace_size, workspace)


def params_for(cu_seqlens_host, hq, hkv, d, dp, top_k, **kw):
    lens = [int(b) - int(a) for a, b in zip(cu_seqlens_host[:-1], cu_seqlens_host[1:])]
    return make_params(int(cu_seqlens_host[-1]), len(lens), max(lens) if lens else 0, hq, hkv, d,
                       dp, top_k, **kw)


def workspace_bytes(params) -> int:
    return max(msa_select_workspace_size(params), msa_fwd_workspace_size(params),
               msa_bwd_workspace_size(params))


class MSAStep:
    """Holds outputs and workspace for repeated steps at one shape."""

    def __init__(self, params, device="cuda", reuse_lists=True):
        self.params = params
        self.out = allocate_outputs(params, device)
        self.ws = workspace(workspace_bytes(params), device)
        self.reuse_lists = reuse_lists
        self._lists = None  # (cu_seqlens pointer, stream) of the call that built the lists
        self._bwd_params = MsaParams.from_buffer_copy(params)  # params + reuse flag
        self._bwd_params.flags = params.flags | MSA_FLAG_REUSE_REGROUP

    def select(self, inp, stream=None):
        o = self.out
        msa_proxy_select(self.params, inp["cu_seqlens"], inp["q_p"], inp["k_p"], o["sel_idx"],
                         o["sel_score"], o["sel_arg"], o["plse"], o["tie"], self.ws, stream)
        # the call left the block lists of this selection in the workspace
        self._lists = (inp["cu_seqlens"].data_ptr(), stream)

    def forward(self, inp, stream=None):
        o = self.out
        reuse = self.reuse_lists and self._lists == (inp["cu_seqlens"].data_ptr(), stream)
        msa_fwd(self._bwd_params if reuse else self.params, inp["cu_seqlens"], inp["q"], inp["k"],
                inp["v"], o["sel_idx"], o["o"], o["o_res"], o["lse"], o["mass"], self.ws, stream)
        self._lists = (inp["cu_seqlens"].data_ptr(), stream)

    def backward(self, inp, stream=None):
        o = self.out
        reuse = self.reuse_lists and self._lists == (inp["cu_seqlens"].data_ptr(), stream)
        msa_bwd(self._bwd_params if reuse else self.params, inp["cu_seqlens"], inp["q"], inp["k"],
                inp["v"], inp["q_p"], inp["k_p"], o["o"], o["o_res"], o["lse"], o["mass"],
                inp["dO"], o["sel_idx"], o["sel_score"], o["sel_arg"], o["plse"], o["dq"],
                o["dk"], o["dv"], o["dq_p"], o["dk_p"], o["kl_loss"], self.ws, stream)

    def __call__(self, inp, stream=None):
        self.select(inp, stream)
        self.forward(inp, stream)
        self.backward(inp, stream)
        return self.out


class HostInputStep:
    """Training steps whose inputs arrive in, and whose results return to,
    pinned host memory.

    The host-to-device copies run on a copy stream in the order the calls need
    them (cu_seqlens, q_p, k_p for the selection; k, v, q for the forward; dO
    for the backward), and each call waits only for its own inputs, so the
    copies of the later inputs overlap the earlier kernels.  `depth` sets of
    device input buffers and of device outputs rotate between steps: the
    copies of step i overlap the kernels of the steps before it and wait only
    for step i - depth's kernels, the last to read the input set they
    overwrite.

    Results go back on a second copy stream: O (and LSE) as soon as the
    forward has finished, so their copy overlaps the backward; the five
    gradients and the proxy-KL loss after the backward, overlapping the next
    steps.  A step's forward and backward wait only for the copies out of the
    output set they overwrite, made depth steps earlier, so a copy that runs
    slow for a while (host-link copy rates vary) holds the kernels back only
    once it is more than depth - 1 steps behind.  Without `host_out`, only the loss is
    copied back (to `self.loss`).  Read host results after synchronising.
    The host tensors are read and written asynchronously: leave the inputs
    unchanged, and do not read the outputs, until the step's copies have
    finished.
    """

    GROUPS = (("cu_seqlens", "q_p", "k_p"), ("k", "v", "q"), ("dO",))
    FWD_OUT = ("o", "lse")
    BWD_OUT = ("dq", "dk", "dv", "dq_p", "dk_p", "kl_loss")

    def __init__(self, params, like: dict, device="cuda", step: MSAStep | None = None,
                 depth: int = 2):
        """like: tensors with the shapes and dtypes of one step's inputs; step:
        an MSAStep of these params whose workspace (and first output set) to
        use; depth: input and output sets in rotation (at least 1)."""
        if depth < 1:
            raise ValueError("HostInputStep: depth must be at least 1")
        self.step = step if step is not None else MSAStep(params, device)
        self.depth = depth
        names = [n for grp in self.GROUPS for n in grp]
        self.bufs = [{n: torch.empty(like[n].shape, dtype=like[n].dtype, device=device)
                      for n in names} for _ in range(depth)]
        self.outs = [self.step.out] + [allocate_outputs(params, device) for _ in range(depth - 1)]
        self.done = [None] * depth  # kernels of the last step that read input set b
        self.fwd_copied = [None] * depth  # copies of O / gradients out of output set b
        self.bwd_copied = [None] * depth
        self.copy_stream = torch.cuda.Stream(device)
        self.out_stream = torch.cuda.Stream(device)
        self.loss = torch.empty(1, dtype=torch.float64).pin_memory()
        self._n = 0

    def allocate_host_outputs(self) -> dict:
        """Pinned host tensors for every result the step returns."""
        out = self.step.out
        return {n: torch.empty(out[n].shape, dtype=out[n].dtype).pin_memory()
                for n in self.FWD_OUT + self.BWD_OUT}

    def __call__(self, host_inp: dict, loss_out: torch.Tensor | None = None,
                 host_out: dict | None = None) -> dict:
        """Queue one step on the current stream; returns the device outputs
        (valid until the kernels of the step depth calls later overwrite
        them)."""
        for grp in self.GROUPS:
            for n in grp:
                t = host_inp[n]
                if t.is_cuda or not t.is_pinned():
                    raise ValueError(f"HostInputStep: input {n!r} must be a pinned host tensor "
                                     "(pageable memory would make every copy synchronous)")
        if host_out is not None:
            for n in self.FWD_OUT + self.BWD_OUT:
                t = host_out[n]
                if t.is_cuda or not t.is_pinned():
                    raise ValueError(f"HostInputStep: output {n!r} must be a pinned host tensor")
        b = self._n % self.depth
        self._n += 1
        dev, cs, os_ = self.bufs[b], self.copy_stream, self.out_stream
        st = torch.cuda.current_stream(cs.device)
        if self.done[b] is not None:
            cs.wait_event(self.done[b])
        ready = []
        with torch.cuda.stream(cs):
            for grp in self.GROUPS:
                for n in grp:
                    dev[n].copy_(host_inp[n], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                ready.append(ev)
        out = self.outs[b]
        self.step.out = out
        st.wait_event(ready[0])
        self.step.select(dev, st)
        st.wait_event(ready[1])
        if self.fwd_copied[b] is not None:  # this set's O of depth steps ago has left
            st.wait_event(self.fwd_copied[b])
        self.step.forward(dev, st)
        if host_out is not None:
            fwd_done = torch.cuda.Event()
            fwd_done.record(st)
            os_.wait_event(fwd_done)
            with torch.cuda.stream(os_):
                for n in self.FWD_OUT:
                    host_out[n].copy_(out[n], non_blocking=True)
            self.fwd_copied[b] = torch.cuda.Event()
            self.fwd_copied[b].record(os_)
        st.wait_event(ready[2])
        if self.bwd_copied[b] is not None:  # this set's gradients of depth steps ago have left
            st.wait_event(self.bwd_copied[b])
        self.step.backward(dev, st)
        done = torch.cuda.Event()
        done.record(st)
        self.done[b] = done
        if host_out is None:
            (self.loss if loss_out is None else loss_out).copy_(out["kl_loss"], non_blocking=True)
        else:
            os_.wait_event(done)
            with torch.cuda.stream(os_):
                for n in self.BWD_OUT:
                    host_out[n].copy_(out[n], non_blocking=True)
            self.bwd_copied[b] = torch.cuda.Event()
            self.bwd_copied[b].record(os_)
        return out

    def wait_outputs(self, stream=None) -> None:
        """Makes `stream` (default: the current one) wait for the result copies
        queued so far."""
        st = stream if stream is not None else torch.cuda.current_stream(self.out_stream.device)
        for ev in self.fwd_copied + self.bwd_copied:
            if ev is not None:
                st.wait_event(ev)


def run_step(params, inp, device="cuda") -> dict:
    step = MSAStep(params, device)
    out = step(inp)
    torch.cuda.synchronize()
    return out
