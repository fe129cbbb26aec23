"""The autograd front end (msa_attention) returns what the C ABI step returns,
also when two calls run their forwards before their backwards."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _step_outputs(w, dev, **pattern):
    from block_sparse_attention_proxy_gb300.step import MSAStep, params_for

    prm = params_for(dev["cu_seqlens"].tolist(), w.hq, w.hkv, w.d, w.dp, w.top_k, **pattern)
    st = MSAStep(prm)
    st(dev)
    return {k: v.clone() for k, v in st.out.items()}


def _autograd(w, dev, **pattern):
    from block_sparse_attention_proxy_gb300.function import msa_attention

    leaves = {n: dev[n].clone().requires_grad_(True) for n in ("q", "k", "v", "q_p", "k_p")}
    o = msa_attention(leaves["q"], leaves["k"], leaves["v"], leaves["q_p"], leaves["k_p"],
                      dev["cu_seqlens"], w.top_k, **pattern)
    return o, leaves


@pytest.mark.parametrize("pattern", [{}, dict(window=2, dilation=2)], ids=["plain", "window"])
def test_autograd_matches_step(pattern):
    from block_sparse_attention_proxy_gb300.function import last_kl_loss

    w = synth.custom([900, 1300], 8, 2, 128, 64, 4, seed=31, structured=True)
    dev = {k: v.cuda() for k, v in synth.make_inputs(w).items()}
    ref = _step_outputs(w, dev, **pattern)
    o, leaves = _autograd(w, dev, **pattern)
    assert torch.equal(o, ref["o"])
    o.backward(dev["dO"])
    for n, g in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("q_p", "dq_p"), ("k_p", "dk_p")):
        assert torch.equal(leaves[n].grad, ref[g].to(leaves[n].grad.dtype)), n
    assert torch.equal(last_kl_loss(), ref["kl_loss"])


def test_two_calls_forward_then_backward():
    w1 = synth.custom([1500], 4, 1, 64, 32, 3, seed=41)
    w2 = synth.custom([700, 800], 4, 1, 64, 32, 3, seed=42)
    d1 = {k: v.cuda() for k, v in synth.make_inputs(w1).items()}
    d2 = {k: v.cuda() for k, v in synth.make_inputs(w2).items()}
    r1, r2 = _step_outputs(w1, d1), _step_outputs(w2, d2)
    o1, l1 = _autograd(w1, d1)
    o2, l2 = _autograd(w2, d2)
    (o1.float() * d1["dO"].float()).sum().add((o2.float() * d2["dO"].float()).sum()).backward()
    for leaves, ref in ((l1, r1), (l2, r2)):
        for n, g in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("q_p", "dq_p"), ("k_p", "dk_p")):
            got = leaves[n].grad.float()
            want = ref[g].to(leaves[n].grad.dtype).float()
            assert torch.allclose(got, want, rtol=1e-2, atol=1e-2), n
