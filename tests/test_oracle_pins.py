"""Pins for the CPU fp64 oracle: each test checks it against something other
than itself (a library routine, brute force, finite differences, autograd,
closed forms, invariants), chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them."""
import itertools
import math

import numpy as np
import pytest
import torch

import synth
from oracle import OracleParams, msa_reference, row_reference, select_from_pooled
from oracle.msa_oracle import mask_pair_count, pooled_proxy_scores


def _inputs(doc_lengths, hq, hkv, d, dp, seed, dtype=torch.float64, structured=False):
    w = synth.custom(doc_lengths, hq, hkv, d, dp, top_k=2, seed=seed, structured=structured)
    return synth.make_inputs(w, device="cpu", dtype=dtype)


def _prm(hq, hkv, d, dp, k, block):
    return OracleParams(hq=hq, hkv=hkv, d=d, dp=dp, top_k=k, block=block)


# ---------------------------------------------------------------------------
# dense limit: k covering every block is dense causal attention (torch SDPA)
# ---------------------------------------------------------------------------
def _sdpa_dense(inp, hq, hkv):
    """Dense causal GQA attention per document with torch's own SDPA (float64 CPU),
    outputs and gradients of sum(O * dO)."""
    G = hq // hkv
    cu = inp["cu_seqlens"].tolist()
    outs, dqs, dks, dvs = [], [], [], []
    for a, b in zip(cu[:-1], cu[1:]):
        q = inp["q"][a:b].double().transpose(0, 1).clone().requires_grad_(True)  # [H, L, d]
        k = inp["k"][a:b].double().transpose(0, 1).clone().requires_grad_(True)
        v = inp["v"][a:b].double().transpose(0, 1).clone().requires_grad_(True)
        kk = k.repeat_interleave(G, dim=0)
        vv = v.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True, scale=1.0)
        (o * inp["dO"][a:b].double().transpose(0, 1)).sum().backward()
        outs.append(o.detach().transpose(0, 1))
        dqs.append(q.grad.transpose(0, 1))
        dks.append(k.grad.transpose(0, 1))
        dvs.append(v.grad.transpose(0, 1))
    return [torch.cat(x).numpy() for x in (outs, dqs, dks, dvs)]


@pytest.mark.parametrize("block", [16, 128])
def test_dense_limit_equals_sdpa(block):
    hq, hkv, d, dp = 4, 2, 16, 8
    inp = _inputs([300, 517, 1], hq, hkv, d, dp, seed=3)
    nb = (517 + block - 1) // block
    prm = _prm(hq, hkv, d, dp, k=nb + 2, block=block)
    ref = msa_reference(inp, prm)
    o, dq, dk, dv = _sdpa_dense(inp, hq, hkv)
    np.testing.assert_allclose(ref["o"], o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ref["dq"], dq, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(ref["dk"], dk, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(ref["dv"], dv, rtol=1e-9, atol=1e-11)


def test_rows_with_few_blocks_are_dense():
    """A row whose block index j <= k-1 keeps every earlier block: dense causal."""
    hq, hkv, d, dp, block, k = 2, 1, 8, 4, 16, 3
    inp = _inputs([200], hq, hkv, d, dp, seed=5)
    ref = msa_reference(inp, _prm(hq, hkv, d, dp, k, block))
    o = _sdpa_dense(inp, hq, hkv)[0]
    rows = np.arange(200) // block <= k - 1
    np.testing.assert_allclose(ref["o"][rows], o[rows], rtol=1e-10, atol=1e-12)
    assert np.abs(ref["o"][~rows] - o[~rows]).max() > 1e-3  # sparse rows differ


# ---------------------------------------------------------------------------
# max-pool and selection
# ---------------------------------------------------------------------------
def test_pooled_scores_brute_force_loops():
    """Max-pool and lowest-index argmax against explicit Python loops over keys."""
    hq, hkv, d, dp, block = 2, 2, 4, 3, 8
    inp = _inputs([37], hq, hkv, d, dp, seed=7)
    prm = _prm(hq, hkv, d, dp, 2, block)
    qp = inp["q_p"].double().numpy()
    kp = inp["k_p"].double().numpy()
    rows = np.arange(37)
    S, A = pooled_proxy_scores(qp, kp, rows, prm)
    for i in range(37):
        for g in range(hkv):
            for b in range(5):
                best, arg = -math.inf, -1
                for key in range(b * block, min((b + 1) * block, 37)):
                    if key > i:
                        break
                    s = sum(qp[i, g, c] * kp[key, g, c] for c in range(dp))
                    if s > best:
                        best, arg = s, key - b * block
                if arg < 0:
                    assert S[i, g, b] == -math.inf and A[i, g, b] == -1
                else:
                    assert abs(S[i, g, b] - best) < 1e-12 and A[i, g, b] == arg


def test_pooled_argmax_prefers_lowest_key_on_exact_tie():
    prm = _prm(1, 1, 1, 1, 2, 4)
    qp = np.ones((8, 1, 1))
    kp = np.array([0.0, 2.0, 1.0, 2.0, 3.0, 3.0, 3.0, -1.0]).reshape(8, 1, 1)
    S, A = pooled_proxy_scores(qp, kp, np.array([7]), prm)
    assert S[0, 0, 0] == 2.0 and A[0, 0, 0] == 1
    assert S[0, 0, 1] == 3.0 and A[0, 0, 1] == 0


@pytest.mark.parametrize("seed", range(6))
def test_selection_matches_brute_force_subsets(seed):
    """Top-(k-1) by score equals the (k-1)-subset of earlier blocks with the
    largest score sum (distinct scores), plus the diagonal."""
    rng = np.random.default_rng(seed)
    for j in range(0, 11):
        for k in (1, 2, 3, 4, 6):
            S = rng.normal(size=j + 1)
            sel, gap = select_from_pooled(S, j, k)
            if j <= k - 1:
                want = list(range(j))
            else:
                want = max(itertools.combinations(range(j), k - 1), key=lambda c: sum(S[list(c)]))
                want = sorted(want)
                srt = np.sort(S[:j])[::-1]
                assert abs(gap - (srt[k - 2] - srt[k - 1])) < 1e-15 if k >= 2 else True
            assert sel[: len(want) + 1] == sorted(want) + [j]
            assert sel[len(want) + 1:] == [-1] * (k - len(want) - 1)


def test_selection_ties_go_to_lower_block():
    # scores of blocks 0..4; the diagonal (5) is not ranked
    S = np.array([1.0, 2.0, 2.0, 2.0, 0.0, 9.0])
    assert select_from_pooled(S, 5, 3)[0] == [1, 2, 5]
    assert select_from_pooled(S, 5, 4)[0] == [1, 2, 3, 5]
    assert select_from_pooled(S, 5, 3)[1] == 0.0  # (k-1)-th and k-th best are tied


# ---------------------------------------------------------------------------
# block pattern: an always-kept window of w blocks spaced s apart
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_window_selection_matches_brute_force_subsets(seed):
    """With a window (w, s), the selection is, among the min(j, k-1)-subsets of
    earlier blocks that hold every block at distance s*u (u = 1..w) behind j,
    the one with the largest score sum (distinct scores), plus the diagonal."""
    rng = np.random.default_rng(100 + seed)
    for j in range(0, 12):
        for k in (2, 3, 4, 6):
            for w in range(0, k):
                for s in (1, 2, 3):
                    S = rng.normal(size=j + 1)
                    sel, gap = select_from_pooled(S, j, k, window=w, dilation=s)
                    must = {b for b in range(j) if (j - b) % s == 0 and (j - b) // s <= w}
                    size = min(j, k - 1)
                    subsets = [c for c in itertools.combinations(range(j), size) if must <= set(c)]
                    want = sorted(max(subsets, key=lambda c: sum(S[list(c)])))
                    assert sel == want + [j] + [-1] * (k - 1 - size), (j, k, w, s)
                    free = sorted((S[b] for b in range(j) if b not in must), reverse=True)
                    nfree = size - len(must)
                    if nfree == 0 or len(free) <= nfree:
                        assert gap == math.inf
                    else:
                        assert abs(gap - (free[nfree - 1] - free[nfree])) < 1e-15


def test_window_must_fit_in_top_k():
    with pytest.raises(ValueError):
        select_from_pooled(np.zeros(8), 7, 3, window=3, dilation=1)
    # a window reaching past the document start keeps only the blocks that exist
    assert select_from_pooled(np.zeros(8), 7, 3, window=2, dilation=5)[0] == [0, 2, 7]


def _sdpa_local(inp, hq, hkv, block, nblocks):
    """Causal GQA attention restricted to keys in the last `nblocks` blocks of
    the query (its own included), per document, with torch's SDPA and an
    explicit boolean mask (float64 CPU); outputs and gradients of sum(O * dO)."""
    G = hq // hkv
    cu = inp["cu_seqlens"].tolist()
    res = [[], [], [], []]
    for a, b in zip(cu[:-1], cu[1:]):
        L = b - a
        pos = torch.arange(L)
        keep = (pos[None, :] <= pos[:, None]) & (pos[None, :] // block > pos[:, None] // block - nblocks)
        q = inp["q"][a:b].double().transpose(0, 1).clone().requires_grad_(True)
        k = inp["k"][a:b].double().transpose(0, 1).clone().requires_grad_(True)
        v = inp["v"][a:b].double().transpose(0, 1).clone().requires_grad_(True)
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k.repeat_interleave(G, dim=0), v.repeat_interleave(G, dim=0), attn_mask=keep,
            scale=1.0)
        (o * inp["dO"][a:b].double().transpose(0, 1)).sum().backward()
        for lst, x in zip(res, (o.detach(), q.grad, k.grad, v.grad)):
            lst.append(x.transpose(0, 1))
    return [torch.cat(x).numpy() for x in res]


def test_full_window_is_sliding_window_attention():
    """w = k-1, s = 1 keeps the last k blocks whatever the proxy says: the
    attention is sliding-window attention over k blocks."""
    hq, hkv, d, dp, block, k = 4, 2, 8, 4, 16, 3
    inp = _inputs([150, 77, 16], hq, hkv, d, dp, seed=21)
    prm = OracleParams(hq=hq, hkv=hkv, d=d, dp=dp, top_k=k, block=block, window=k - 1)
    ref = msa_reference(inp, prm)
    o, dq, dk, dv = _sdpa_local(inp, hq, hkv, block, k)
    np.testing.assert_allclose(ref["o"], o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ref["dq"], dq, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(ref["dk"], dk, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(ref["dv"], dv, rtol=1e-9, atol=1e-11)


# ---------------------------------------------------------------------------
# gradients: central finite differences of the forward (fp64)
# ---------------------------------------------------------------------------
def _loss(inp, prm, sel, arg, mass0):
    out = msa_reference(inp, prm, sel_override=sel, arg_override=arg, with_grads=False)
    main = float(np.sum(out["o"] * inp["dO"].numpy()))
    valid = sel >= 0
    with np.errstate(divide="ignore", invalid="ignore"):
        kl = np.where(valid & (mass0 > 0), mass0 * (np.log(mass0) - np.log(out["p"])), 0.0)
    return main + prm.kl_weight * float(kl.sum())


def test_gradients_match_finite_differences():
    hq, hkv, d, dp, block, k = 4, 2, 16, 8, 128, 3
    inp = _inputs([640], hq, hkv, d, dp, seed=11)
    prm = _prm(hq, hkv, d, dp, k, block)
    prm.kl_weight = 0.7
    ref = msa_reference(inp, prm)
    sel, arg, mass0 = ref["sel_idx"], ref["sel_arg"], ref["mass"]
    rng = np.random.default_rng(0)
    eps = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("q_p", "dq_p"), ("k_p", "dk_p")):
        for _ in range(3):
            u = rng.normal(size=inp[name].shape)
            plus = dict(inp)
            minus = dict(inp)
            plus[name] = inp[name] + eps * torch.from_numpy(u)
            minus[name] = inp[name] - eps * torch.from_numpy(u)
            fd = (_loss(plus, prm, sel, arg, mass0) - _loss(minus, prm, sel, arg, mass0)) / (2 * eps)
            an = float(np.sum(ref[gname] * u))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


# ---------------------------------------------------------------------------
# gradients: torch.autograd through an independently written dense formulation
# ---------------------------------------------------------------------------
def _autograd_step(inp, sel, prm):
    """Dense masked softmax with the block mask from `sel`, block max via torch.max,
    KL(m.detach() || p); gradients by autograd."""
    B, G = prm.block, prm.group
    T = inp["q"].shape[0]
    t = {n: inp[n].double().clone().requires_grad_(True) for n in ("q", "k", "v", "q_p", "k_p")}
    dO = inp["dO"].double()
    total = 0.0
    cu = inp["cu_seqlens"].tolist()
    for a, b in zip(cu[:-1], cu[1:]):
        L = b - a
        NB = (L + B - 1) // B
        pos = torch.arange(L)
        causal = pos[None, :] <= pos[:, None]
        for g in range(prm.hkv):
            chosen = torch.zeros(L, NB, dtype=torch.bool)
            sl = torch.from_numpy(sel[a:b, g])
            for s in range(prm.top_k):
                ok = sl[:, s] >= 0
                chosen[pos[ok], sl[ok, s]] = True
            mask = causal & chosen[:, pos // B]
            mass_b = torch.zeros(L, NB, dtype=torch.float64)
            for hh in range(G):
                h = g * G + hh
                z = t["q"][a:b, h] @ t["k"][a:b, g].T * prm.softmax_scale
                z = z.masked_fill(~mask, float("-inf"))
                P = torch.softmax(z, dim=1)
                o = P @ t["v"][a:b, g]
                total = total + (o * dO[a:b, h]).sum()
                pad = torch.zeros(L, NB * B, dtype=torch.float64)
                pad[:, :L] = P.detach()
                mass_b = mass_b + pad.reshape(L, NB, B).sum(2) / G
            s = (t["q_p"][a:b, g] @ t["k_p"][a:b, g].T) * prm.proxy_scale
            s = s.masked_fill(~causal, float("-inf"))
            spad = torch.full((L, NB * B), float("-inf"), dtype=torch.float64)
            spad[:, :L] = s
            S = spad.reshape(L, NB, B).max(dim=2).values  # [L, NB]
            S = S.masked_fill(~chosen, float("-inf"))
            logp = torch.log_softmax(S, dim=1)
            m = mass_b.masked_fill(~chosen, 0.0)
            kl = torch.where(m > 0, m * (torch.log(m.clamp_min(1e-300)) - logp),
                             torch.zeros_like(m)).sum()
            total = total + prm.kl_weight * kl
    total.backward()
    return {("d" + n): t[n].grad.numpy() for n in t}, float(total)


@pytest.mark.parametrize("window,dilation", [(0, 1), (1, 2)])
def test_gradients_match_autograd(window, dilation):
    hq, hkv, d, dp, block, k = 4, 2, 8, 4, 16, 3
    inp = _inputs([90, 161], hq, hkv, d, dp, seed=13)
    prm = OracleParams(hq=hq, hkv=hkv, d=d, dp=dp, top_k=k, block=block, window=window,
                       dilation=dilation)
    ref = msa_reference(inp, prm)
    grads, _ = _autograd_step(inp, ref["sel_idx"], prm)
    for n in ("dq", "dk", "dv", "dq_p", "dk_p"):
        np.testing.assert_allclose(ref[n], grads[n], rtol=1e-9, atol=1e-11, err_msg=n)


# ---------------------------------------------------------------------------
# invariants and closed-form special cases
# ---------------------------------------------------------------------------
def test_invariants():
    hq, hkv, d, dp, block, k = 6, 2, 8, 4, 16, 4
    inp = _inputs([150, 33, 97], hq, hkv, d, dp, seed=17)
    prm = _prm(hq, hkv, d, dp, k, block)
    ref = msa_reference(inp, prm)
    valid = ref["sel_idx"] >= 0
    np.testing.assert_allclose(ref["p"].sum(2), 1.0, atol=1e-12)
    np.testing.assert_allclose(ref["mass"].sum(2), 1.0, atol=1e-12)
    gb = np.where(valid, ref["p"] - ref["mass"], 0.0)
    np.testing.assert_allclose(gb.sum(2), 0.0, atol=1e-12)
    assert (ref["kl"] >= -1e-14).all()
    # rows in their document's first block: one block, p = m = 1, no proxy gradient
    cu = inp["cu_seqlens"].tolist()
    first = np.concatenate([np.arange(a, min(b, a + block)) for a, b in zip(cu[:-1], cu[1:])])
    np.testing.assert_allclose(ref["kl"][first], 0.0, atol=1e-14)
    np.testing.assert_allclose(ref["dq_p"][first], 0.0, atol=1e-14)
    # rows of P sum to one, so per document sum_keys dv = sum of the group's dO,
    # and sum_keys dS = 0 gives sum_keys dk = 0
    G = prm.group
    dO = inp["dO"].double().numpy()
    for a, b in zip(cu[:-1], cu[1:]):
        for g in range(hkv):
            np.testing.assert_allclose(ref["dv"][a:b, g].sum(0), dO[a:b, g * G:(g + 1) * G].sum((0, 1)),
                                       atol=1e-10)
            np.testing.assert_allclose(ref["dk"][a:b, g].sum(0), 0.0, atol=1e-10)
    # the effective pair count equals the mask size counted key by key from the
    # selection the reference attended over (every selected block, keys <= i)
    sel = ref["sel_idx"]
    counted = 0
    for a, b in zip(cu[:-1], cu[1:]):
        for i in range(b - a):
            for blk in sel[a + i, 0]:
                if blk >= 0:
                    counted += sum(1 for key in range(blk * block, (blk + 1) * block) if key <= i)
    assert mask_pair_count(inp["cu_seqlens"], prm) == counted * hq


def test_uniform_scores_closed_form():
    """q = 0 and q_p = 0: attention is uniform over the mask, p is uniform over the
    selection (ties -> the k-1 lowest earlier blocks), m_b = |b ∩ M| / |M|,
    KL = sum_b m_b log(m_b n)."""
    hq, hkv, d, dp, block, k = 2, 1, 4, 2, 4, 3
    L = 14
    inp = _inputs([L], hq, hkv, d, dp, seed=19)
    inp["q"] = torch.zeros_like(inp["q"])
    inp["q_p"] = torch.zeros_like(inp["q_p"])
    prm = _prm(hq, hkv, d, dp, k, block)
    ref = msa_reference(inp, prm)
    v = inp["v"].double().numpy()[:, 0]
    for i in range(L):
        j, r = divmod(i, block)
        blocks = list(range(min(j, k - 1))) + [j]
        assert list(ref["sel_idx"][i, 0, : len(blocks)]) == blocks
        keys = [key for b in blocks for key in range(b * block, min((b + 1) * block, i + 1))]
        np.testing.assert_allclose(ref["o"][i, 0], v[keys].mean(0), atol=1e-14)
        np.testing.assert_allclose(ref["lse"][i], math.log(len(keys)), atol=1e-14)
        m = np.array([len([x for x in keys if x // block == b]) / len(keys) for b in blocks])
        np.testing.assert_allclose(ref["mass"][i, 0, : len(blocks)], m, atol=1e-14)
        np.testing.assert_allclose(ref["p"][i, 0, : len(blocks)], 1.0 / len(blocks), atol=1e-14)
        np.testing.assert_allclose(ref["kl"][i, 0], float(np.sum(m * np.log(m * len(blocks)))),
                                   atol=1e-13)


def test_single_token_document():
    hq, hkv, d, dp = 4, 2, 8, 4
    inp = _inputs([5, 1, 3], hq, hkv, d, dp, seed=23)
    ref = msa_reference(inp, _prm(hq, hkv, d, dp, 2, 16))
    t = 5
    for h in range(hq):
        g = h // 2
        np.testing.assert_allclose(ref["o"][t, h], inp["v"][t, g].double().numpy(), atol=1e-15)
        np.testing.assert_allclose(ref["lse"][t, h],
                                   float(inp["q"][t, h].double() @ inp["k"][t, g].double()), atol=1e-14)
    assert list(ref["sel_idx"][t, 0]) == [0, -1]
    np.testing.assert_allclose(ref["kl"][t], 0.0)
    np.testing.assert_allclose(ref["dq"][t], 0.0, atol=1e-15)  # one key: dS = 0


def test_group_of_one_is_per_head_attention():
    """With G = 1 (MHA) each head is an independent single-head problem."""
    hq = hkv = 2
    d, dp, block, k = 8, 4, 16, 2
    inp = _inputs([70], hq, hkv, d, dp, seed=29)
    both = msa_reference(inp, _prm(hq, hkv, d, dp, k, block))
    for h in range(2):
        one = {n: (x[:, h:h + 1] if x.dim() == 3 else x) for n, x in inp.items()}
        r = msa_reference(one, _prm(1, 1, d, dp, k, block))
        for n in ("o", "dq", "dk", "dv", "dq_p", "dk_p"):
            np.testing.assert_allclose(both[n][:, h:h + 1], r[n], atol=1e-13, err_msg=n)
        np.testing.assert_allclose(both["kl"][:, h:h + 1], r["kl"], atol=1e-13)


def test_zero_proxy_keys_give_uniform_proxy():
    hq, hkv, d, dp, block, k = 2, 1, 8, 4, 16, 3
    inp = _inputs([90], hq, hkv, d, dp, seed=31)
    inp["k_p"] = torch.zeros_like(inp["k_p"])
    ref = msa_reference(inp, _prm(hq, hkv, d, dp, k, block))
    n = (ref["sel_idx"] >= 0).sum(2)
    np.testing.assert_allclose(ref["p"].sum(2), 1.0)
    np.testing.assert_allclose(np.where(ref["sel_idx"] >= 0, ref["p"], 1.0 / n[..., None]),
                               (1.0 / n)[..., None] * np.ones_like(ref["p"]), atol=1e-15)
    np.testing.assert_allclose(ref["dq_p"], 0.0, atol=1e-15)  # k_p = 0


# ---------------------------------------------------------------------------
# the one-row reference agrees with the whole-document reference
# ---------------------------------------------------------------------------
def test_row_reference_matches_full():
    hq, hkv, d, dp, block, k = 4, 2, 16, 8, 16, 3
    inp = _inputs([100, 143], hq, hkv, d, dp, seed=37, structured=True)
    prm = _prm(hq, hkv, d, dp, k, block)
    full = msa_reference(inp, prm)
    dk = np.zeros_like(full["dk"])
    dv = np.zeros_like(full["dv"])
    dkp = np.zeros_like(full["dk_p"])
    for t in range(243):
        r = row_reference(inp, prm, t, contributions=True)
        assert (r["sel"] == full["sel_idx"][t]).all()
        for n in ("sel_score", "plse", "o", "lse", "mass", "p", "kl", "dq", "dq_p"):
            key = {"o": "o"}.get(n, n)
            np.testing.assert_allclose(r[n], full[key][t], atol=1e-12, err_msg=n)
        for c in r["contrib"]:
            np.add.at(dk[:, c["g"]], c["keys"], c["dk"])
            np.add.at(dv[:, c["g"]], c["keys"], c["dv"])
            np.add.at(dkp[:, c["g"]], c["dkp_keys"], c["dkp"])
    np.testing.assert_allclose(dk, full["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, full["dv"], atol=1e-12)
    np.testing.assert_allclose(dkp, full["dk_p"], atol=1e-12)
