"""Failure detection on the GPU without a fault: a bounded wait that runs out.

MSA_FLAG_TEST_STALL_SELECT makes the selection kernel withhold the load its
MMA warp waits for.  After the bounded-wait limit (about half a second of SM
cycles) each CTA records MSA_ERR_TIMEOUT with the site of the wait, lets its
own copies land, frees its tensor memory and returns without writing its
outputs.  The test reads the status word and its site, checks that the
outputs of the earlier call are untouched, and that the next call without the
flag is correct (bit for bit a repeat of a clean step) and leaves status 0.
"""
import time

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

MSA_ERR_TIMEOUT = 5
KERNEL_SELECT = 1
# barriers of the selection kernel a stalled CTA can give up on: the query
# tile (MMA warp), the k_p ring stages (producer) and the two score
# accumulators (epilogue)
SELECT_WAITS = {0, 7, 8, 9, 10, 11, 12, 13, 14}


def test_select_wait_that_runs_out_reports_timeout_and_next_call_is_clean():
    import block_sparse_attention_proxy_gb300 as m
    from block_sparse_attention_proxy_gb300.step import MSAStep, params_for

    w = synth.workload("tiny")
    dev = {k: v.cuda() for k, v in synth.make_inputs(w).items()}
    prm = params_for(dev["cu_seqlens"].tolist(), w.hq, w.hkv, w.d, w.dp, w.top_k)
    first = MSAStep(prm)
    first(dev)
    torch.cuda.synchronize()
    assert m.msa_get_device_status() == 0
    want = {k: v.clone() for k, v in first.out.items()}

    stall = m.MsaParams.from_buffer_copy(prm)
    stall.flags |= m.MSA_FLAG_TEST_STALL_SELECT
    o = first.out
    t0 = time.perf_counter()
    m.msa_proxy_select(stall, dev["cu_seqlens"], dev["q_p"], dev["k_p"], o["sel_idx"],
                       o["sel_score"], o["sel_arg"], o["plse"], o["tie"], first.ws)
    status = m.msa_get_device_status()
    seconds = time.perf_counter() - t0
    word = m.msa_last_status_word()
    assert status == MSA_ERR_TIMEOUT, (status, hex(word))
    assert (word >> 8) & 0xF == KERNEL_SELECT, hex(word)
    assert (word >> 12) & 0xFF in SELECT_WAITS, hex(word)
    assert (word >> 20) < 4096, hex(word)
    assert seconds < 60, seconds
    for n in ("sel_idx", "sel_score", "sel_arg", "plse", "tie"):
        assert torch.equal(o[n], want[n]), n
    assert m.msa_get_device_status() == 0  # read-and-reset left it clean

    step = MSAStep(prm)
    step(dev)
    torch.cuda.synchronize()
    assert m.msa_get_device_status() == 0
    for n, v in want.items():
        assert torch.equal(step.out[n], v), n
