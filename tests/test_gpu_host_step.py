"""HostInputStep: inputs in pinned host memory, copied on a copy stream that
overlaps the kernels (within a step, and across steps through rotating device
buffer and output sets).  Steps queued back to back, with no synchronisation in
between, must return bit for bit what MSAStep returns on device inputs; the
fourth step reuses the first buffer set, so a copy that overtook the kernels
still reading that set would show."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

SHAPE = ([2500, 700, 1300], 8, 2, 128, 64, 5)


def test_host_input_steps_match_device_steps():
    from block_sparse_attention_proxy_gb300 import msa_get_device_status
    from block_sparse_attention_proxy_gb300.step import HostInputStep, MSAStep, params_for

    lens, hq, hkv, d, dp, k = SHAPE
    sets = [synth.make_inputs(synth.custom(lens, hq, hkv, d, dp, k, seed=60 + i, structured=True))
            for i in range(3)]
    prm = params_for(sets[0]["cu_seqlens"].tolist(), hq, hkv, d, dp, k)

    ref = []
    st = MSAStep(prm)
    for inp in sets:
        out = st({n: v.cuda() for n, v in inp.items()})
        torch.cuda.synchronize()
        ref.append({n: v.clone() for n, v in out.items()})
    assert msa_get_device_status() == 0

    host = [{n: v.pin_memory() for n, v in inp.items()} for inp in sets]
    hs = HostInputStep(prm, sets[0])
    order = [0, 1, 2, 0]
    losses = [torch.empty(1, dtype=torch.float64).pin_memory() for _ in order]
    for j, i in enumerate(order):
        out = hs(host[i], loss_out=losses[j])
    torch.cuda.synchronize()
    assert msa_get_device_status() == 0
    for j, i in enumerate(order):
        assert torch.equal(losses[j], ref[i]["kl_loss"].cpu()), (j, i)
    for n in ("o", "lse", "dq", "dk", "dv", "dq_p", "dk_p", "sel_idx"):
        assert torch.equal(out[n], ref[order[-1]][n]), n


def test_host_input_step_rejects_pageable_inputs():
    from block_sparse_attention_proxy_gb300.step import HostInputStep, params_for

    lens, hq, hkv, d, dp, k = SHAPE
    inp = synth.make_inputs(synth.custom(lens, hq, hkv, d, dp, k, seed=60))
    hs = HostInputStep(params_for(inp["cu_seqlens"].tolist(), hq, hkv, d, dp, k), inp)
    with pytest.raises(ValueError):
        hs(inp)  # pageable CPU tensors


@pytest.mark.parametrize("depth", [1, 2, 3])
def test_host_outputs_of_every_step_match_device_steps(depth):
    """With host_out, O, LSE, the five gradients and the loss of every step
    come back to pinned host memory while later steps run; each step's copy
    must hold that step's results bit for bit (a copy that a later step's
    kernels overtook would hold the later step's values).  depth input and
    output sets rotate; five steps wrap around each of them."""
    from block_sparse_attention_proxy_gb300 import msa_get_device_status
    from block_sparse_attention_proxy_gb300.step import HostInputStep, MSAStep, params_for

    lens, hq, hkv, d, dp, k = SHAPE
    sets = [synth.make_inputs(synth.custom(lens, hq, hkv, d, dp, k, seed=70 + i, structured=True))
            for i in range(3)]
    prm = params_for(sets[0]["cu_seqlens"].tolist(), hq, hkv, d, dp, k)
    ref = []
    st = MSAStep(prm)
    for inp in sets:
        out = st({n: v.cuda() for n, v in inp.items()})
        torch.cuda.synchronize()
        ref.append({n: v.cpu() for n, v in out.items()})
    host = [{n: v.pin_memory() for n, v in inp.items()} for inp in sets]
    hs = HostInputStep(prm, sets[0], depth=depth)
    order = [0, 1, 2, 0, 1]
    outs = [hs.allocate_host_outputs() for _ in order]
    for j, i in enumerate(order):
        hs(host[i], host_out=outs[j])
    hs.wait_outputs()
    torch.cuda.synchronize()
    assert msa_get_device_status() == 0
    for j, i in enumerate(order):
        for n in HostInputStep.FWD_OUT + HostInputStep.BWD_OUT:
            assert torch.equal(outs[j][n], ref[i][n]), (j, i, n)
