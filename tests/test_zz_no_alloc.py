"""msa_proxy_select_noalloc against msa_proxy_select.

The no-allocation entry point exists for host programs that cannot give the
library a device buffer (their device memory is owned by another allocator,
or the calling path may not run cudaMalloc); its scratch is a static device
array inside the library.  It must produce exactly what the workspace entry
point produces, call after call: the second call below runs a batch with a
different document count, so stale contents of the shared array from the
first call would show.  This file is collected last so that a failure here
leaves every other test already run.
"""
import ctypes

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _select(m, prm, dev, noalloc):
    out = m.allocate_outputs(prm)
    if noalloc:
        m.msa_proxy_select_noalloc(prm, dev["cu_seqlens"], dev["q_p"], dev["k_p"], out["sel_idx"],
                                   out["sel_score"], out["sel_arg"], out["plse"], out["tie"])
    else:
        ws = m.workspace(m.msa_select_workspace_size(prm))
        m.msa_proxy_select(prm, dev["cu_seqlens"], dev["q_p"], dev["k_p"], out["sel_idx"],
                           out["sel_score"], out["sel_arg"], out["plse"], out["tie"], ws)
    torch.cuda.synchronize()
    assert m.msa_get_device_status() == 0
    return out


def test_noalloc_select_matches_workspace_select_twice():
    import block_sparse_attention_proxy_gb300 as m
    from block_sparse_attention_proxy_gb300.step import params_for

    cases = [(synth.custom([700, 1, 1500, 333], 8, 2, 128, 64, 5, seed=41, structured=True), {}),
             (synth.custom([2048], 4, 1, 64, 32, 4, seed=42), {}),
             (synth.custom([3000, 500], 8, 2, 128, 64, 6, seed=43), dict(window=3, dilation=2))]
    for w, pattern in cases:
        inp = synth.make_inputs(w)
        dev = {k: v.cuda() for k, v in inp.items()}
        prm = params_for(inp["cu_seqlens"].tolist(), w.hq, w.hkv, w.d, w.dp, w.top_k, **pattern)
        ref = _select(m, prm, dev, noalloc=False)
        got = _select(m, prm, dev, noalloc=True)
        for name in ("sel_idx", "sel_arg", "tie"):
            assert torch.equal(got[name], ref[name]), name
        for name in ("sel_score", "plse"):
            torch.testing.assert_close(got[name], ref[name], rtol=0, atol=1e-6)


def test_noalloc_rejects_batches_beyond_its_scratch():
    import block_sparse_attention_proxy_gb300 as m

    prm = m.make_params(16383 * 2, 16383, 2, 4, 1, 64, 32, 4)
    lib = m.load()
    p = ctypes.c_void_p(0x1000)
    rc = lib.msa_proxy_select_noalloc(ctypes.byref(prm), p, p, p, p, p, p, p, p, None)
    assert rc == 3  # MSA_ERR_WORKSPACE: more documents than the static scratch holds
