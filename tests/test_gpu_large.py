"""Full-size parity for the bench workloads (128k, 512k and 1M tokens; the
512k and 1M steps run in query chunks), in the launch configuration bench.py times
(one MSAStep: select, forward, backward through the C ABI).

The oracle cannot run every row of a 128k-token step, so it checks:
  * 256 seeded query rows (rows 0 and T-1 included): selection (exact outside
    the 1e-3 tie band), tie flag, argmax offsets, O, LSE, target mass, dQ and
    dq_p of every head/group;
  * whole KV blocks for dK, dV and dk_p, at least one in every KV group: every
    token whose selection contains the block (read from the GPU's sel_idx,
    whose rows are themselves checked against the oracle here) is recomputed
    by the oracle and its contributions summed.  Two blocks each in the first
    and last group sit in the middle and at three quarters of the sequence
    (long chooser lists); the other groups take one seeded block among the
    last 64 (short lists, so the oracle stays within seconds per block).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import OracleParams, row_reference
from parity import assert_close, check_argmax_row, check_selection_row, check_tie_flags

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _host_inputs(inp):
    cpu = {k: v.to("cpu") for k, v in inp.items()}
    # k_p prefixes are read by every sampled row: upcast once (exact)
    cpu["k_p"] = cpu["k_p"].double().numpy()
    return cpu


@pytest.mark.parametrize("name,window,dilation",
                         [("128k", 0, 1), ("512k", 0, 1), ("1m", 0, 1), ("128k", 5, 3)],
                         ids=["128k", "512k", "1m", "128k-window5-dilation3"])
def test_full_size_sampled(name, window, dilation):
    import block_sparse_attention_proxy_gb300 as m
    from block_sparse_attention_proxy_gb300.step import MSAStep, params_for

    w = synth.workload(name)
    inp = synth.make_inputs(w, device="cuda")
    prm_c = params_for(inp["cu_seqlens"].tolist(), w.hq, w.hkv, w.d, w.dp, w.top_k,
                       window=window, dilation=dilation)
    step = MSAStep(prm_c)
    step(inp)
    torch.cuda.synchronize()
    assert m.msa_get_device_status() == 0
    g = {k: v.cpu() for k, v in step.out.items()}
    cpu = _host_inputs(inp)
    del inp, step
    torch.cuda.empty_cache()
    prm = OracleParams(w.hq, w.hkv, w.d, w.dp, w.top_k, window=window, dilation=dilation)
    T = w.total_tokens
    sel = g["sel_idx"].numpy()
    arg = g["sel_arg"].numpy()

    # ---- sampled rows ----
    rows = synth.sample_rows(T, 256, w.seed).tolist()
    acc = {n: ([], []) for n in ("o", "lse", "mass", "dq", "dq_p", "sel_score", "plse")}
    tgap, ttie, n_arg = [], [], 0
    for t in rows:
        r = row_reference(cpu, prm, t, sel_override=sel[t], arg_override=arg[t])
        tgap.append(r["gap"])
        ttie.append(g["tie"][t].numpy())
        for gg in range(w.hkv):
            check_selection_row(sel[t, gg], r["sel"][gg], r["pooled"][gg], t // 128, w.top_k,
                                window, dilation)

            def score_of(blk, off, t=t, gg=gg):
                key = blk * 128 + off
                if key > t:  # one document: doc-local = global
                    return -np.inf
                return float(cpu["q_p"][t, gg].double() @ torch.from_numpy(cpu["k_p"][key, gg]))

            n_arg += check_argmax_row(sel[t, gg], arg[t, gg], r["sel"][gg], r["own_arg"][gg],
                                      r["pooled"][gg], score_of)
        acc["o"][0].append(g["o"][t].float().numpy()); acc["o"][1].append(r["o"])
        acc["lse"][0].append(g["lse"][t].numpy()); acc["lse"][1].append(r["lse"])
        acc["mass"][0].append(g["mass"][t].numpy()); acc["mass"][1].append(r["mass"])
        acc["dq"][0].append(g["dq"][t].numpy()); acc["dq"][1].append(r["dq"])
        acc["dq_p"][0].append(g["dq_p"][t].numpy()); acc["dq_p"][1].append(r["dq_p"])
        acc["sel_score"][0].append(g["sel_score"][t].numpy()); acc["sel_score"][1].append(r["sel_score"])
        acc["plse"][0].append(g["plse"][t].numpy()); acc["plse"][1].append(r["plse"])
    check_tie_flags(np.stack(ttie), np.stack(tgap))
    tol = dict(lse=1e-2, mass=5e-3, sel_score=1e-3, plse=1e-3)
    for n, (a, b) in acc.items():
        assert_close(n, np.stack(a), np.stack(b), abs_max=tol.get(n, 2e-2))

    # ---- sampled KV blocks: dK, dV, dk_p ----
    NB = T // 128
    K = w.top_k
    blocks = [(0, NB - 1), (0, NB // 2), (w.hkv - 1, NB - 2), (w.hkv - 1, 3 * NB // 4)]
    rng = np.random.default_rng(w.seed)
    blocks += [(gg, NB - 1 - int(rng.integers(0, 64))) for gg in range(1, w.hkv - 1)]
    for gg, b in blocks:
        off = sel[:, gg, : K - 1]
        choosers = set(np.nonzero((off == b).any(axis=1))[0].tolist())
        choosers |= set(range(b * 128, (b + 1) * 128))
        keys = np.arange(b * 128, (b + 1) * 128)
        dk = np.zeros((128, w.d)); dv = np.zeros((128, w.d)); dkp = np.zeros((128, w.dp))
        for t in sorted(choosers):
            r = row_reference(cpu, prm, t, sel_override=sel[t], arg_override=arg[t],
                              contributions=True, groups=[gg])
            for c in r["contrib"]:
                msk = (c["keys"] >= keys[0]) & (c["keys"] <= keys[-1])
                np.add.at(dk, c["keys"][msk] - keys[0], c["dk"][msk])
                np.add.at(dv, c["keys"][msk] - keys[0], c["dv"][msk])
                mk = (c["dkp_keys"] >= keys[0]) & (c["dkp_keys"] <= keys[-1])
                np.add.at(dkp, c["dkp_keys"][mk] - keys[0], c["dkp"][mk])
        assert_close(f"dk[g{gg},b{b}]", g["dk"][keys, gg].numpy(), dk)
        assert_close(f"dv[g{gg},b{b}]", g["dv"][keys, gg].numpy(), dv)
        assert_close(f"dk_p[g{gg},b{b}]", g["dk_p"][keys, gg].numpy(), dkp)
