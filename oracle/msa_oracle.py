"""Plain, slow fp64 CPU definition of one MSA training step.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg, never by the library.  It shares no code
with the CUDA path.

What is computed, and where it comes from
-----------------------------------------
The pages describe MiniMax Sparse Attention (MSA) training as follows:

* a proxy head scores keys, and KV is chosen in 128-token blocks by the
  *maximum* proxy score inside each block ("Dramatically Speeding Up
  Million-Token Training! ... 'Flash-MSA' ...", ai-minor.com, section "What's
  Happening? News Overview", block-level sparsity bullet; the Flash-MSA summary
  on socker-news.uzaya.net, 要約, "max-pooling を介して");
* important KV is selected in block units ("... 'Flash-MSA' ...", section
  "Terminology Explained", MSA entry);
* attention is grouped-query (GQA) instead of MLA (same page, News Overview);
* the backward passes of the proxy and of the main attention are fused ("...
  'Flash-MSA' ...", section "Why Does This Matter?", fused-backward bullet).

The pages leave the rest open.  This library adopts these definitions (each
listed as a reading in the design notes):

  notation: doc-local position i of token t, block j = i // B, offset r = i % B,
            query head h uses KV group g = h // G with G = Hq / Hkv.
  1. proxy score      s[i,key] = proxy_scale * q_p[t,g] . k_p[key,g], key <= i
  2. block max-pool   S_b = max over keys of block b with key <= i; a_b = the
                      lowest key attaining it (stored as offset in the block)
  3. selection        the diagonal block j is always kept; of b < j keep all if
                      j <= k-1, else the k-1 largest S_b, ties to the lower b.
                      Block pattern (window w, dilation s; w = 0 is the plain
                      rule): the blocks F = {j - s u : 1 <= u <= w, j - s u >= 0}
                      are kept as well, inside the k slots, and the top-k
                      choice fills the other k-1-|F| slots from b < j, b not in F
  4. mask             M[i,key] = key <= i and key // B selected
  5. attention        z = softmax_scale * q[t,h] . k[key,g] on M,
                      LSE = logsumexp z, P = exp(z - LSE), O = sum P v
  6. target mass      m_b = (1/G) sum_{h in g} sum_{key in b, M} P_h   (stop-grad)
  7. proxy dist.      p_b = softmax over selected b of S_b (plse = its logsumexp)
  8. KL               KL_{t,g} = sum_b m_b (log m_b - log p_b), 0 log 0 = 0;
                      L_kl = kl_weight * sum_{t,g} KL_{t,g}
  9. gradients of     L = sum(O * dO) + L_kl, selection and target held fixed:
                      D = rowsum(dO * O), dP = dO v^T, dS = P (dP - D),
                      dq = scale dS k, dk = scale dS^T q, dv = P^T dO (summed
                      over the group's heads);  g_b = kl_weight (p_b - m_b),
                      dq_p = proxy_scale sum_b g_b k_p[a_b],
                      dk_p[a_b] += proxy_scale g_b q_p[t].

Every function below is pinned by tests that do not reuse its code: dense
causal attention when k covers every block, brute-force subset search for the
selection (with and without an always-kept window), sliding-window attention
through torch's SDPA with an explicit mask when the window fills the k slots,
central finite differences and torch.autograd for the gradients, and the
invariants sum p = sum m = 1, sum g = 0, KL >= 0.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

NEG_INF = -np.inf


@dataclasses.dataclass
class OracleParams:
    hq: int
    hkv: int
    d: int
    dp: int
    top_k: int
    block: int = 128
    softmax_scale: float = 1.0
    proxy_scale: float = 1.0
    kl_weight: float = 1.0
    window: int = 0
    dilation: int = 1

    @property
    def group(self) -> int:
        return self.hq // self.hkv


def _f64(x) -> np.ndarray:
    """Exact upcast of a (bf16 / fp32) torch tensor or array to a numpy fp64 array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: only to upcast torch tensors exactly

        return x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        return x.detach().to("cpu").numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def doc_bounds(cu_seqlens):
    cu = _i64(cu_seqlens)
    return [(int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]


def _logsumexp(x: np.ndarray, axis: int) -> np.ndarray:
    m = np.max(x, axis=axis, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    s = np.sum(np.exp(x - m_safe), axis=axis, keepdims=True)
    with np.errstate(divide="ignore"):
        out = np.log(s) + m_safe
    return np.squeeze(out, axis=axis)


# ---------------------------------------------------------------------------
# steps 1-2: proxy scores and block max-pool
# ---------------------------------------------------------------------------
def pooled_proxy_scores(q_p_doc: np.ndarray, k_p_doc: np.ndarray, rows: np.ndarray,
                        prm: OracleParams):
    """Pooled proxy scores for the given doc-local query rows of one document.

    q_p_doc, k_p_doc: [L, Hkv, dp] fp64.  Returns S [R, Hkv, NB] (-inf for
    blocks after the row's own block) and A [R, Hkv, NB] (offset inside the
    block of the lowest key attaining the maximum, -1 where S is -inf).
    """
    L = k_p_doc.shape[0]
    B = prm.block
    NB = (L + B - 1) // B
    R = len(rows)
    S = np.full((R, prm.hkv, NB), NEG_INF)
    A = np.full((R, prm.hkv, NB), -1, dtype=np.int64)
    keys = np.arange(NB * B)
    for g in range(prm.hkv):
        for c0 in range(0, R, 512):
            rr = rows[c0:c0 + 512]
            s = prm.proxy_scale * (q_p_doc[rr, g, :] @ k_p_doc[:, g, :].T)  # [r, L]
            s_pad = np.full((len(rr), NB * B), NEG_INF)
            s_pad[:, :L] = s
            s_pad[keys[None, :] > rr[:, None]] = NEG_INF  # causal: keys <= i only
            blocks = s_pad.reshape(len(rr), NB, B)
            S[c0:c0 + len(rr), g, :] = blocks.max(axis=2)
            arg = blocks.argmax(axis=2)  # first occurrence = lowest key
            arg[~np.isfinite(S[c0:c0 + len(rr), g, :])] = -1
            A[c0:c0 + len(rr), g, :] = arg
    return S, A


# ---------------------------------------------------------------------------
# step 3: top-k selection with the diagonal always kept
# ---------------------------------------------------------------------------
def forced_blocks(j: int, window: int, dilation: int) -> list:
    """The always-kept earlier blocks of block j under a block pattern of
    `window` blocks spaced `dilation` apart: j - dilation * u for u = 1..window,
    those >= 0.  The pattern is configurable by window size and dilation
    ("Flash-MSA: Ein Training mit einer Million Tokens ohne hohe
    Rechenkosten", keelcrux.com, section "Under the hood"); the set itself is
    this library's reading of those two words."""
    return [j - dilation * u for u in range(1, window + 1) if j - dilation * u >= 0]


def select_from_pooled(S_row: np.ndarray, j: int, k: int, window: int = 0, dilation: int = 1):
    """Selection for one (row, group).  S_row holds S_b for b = 0..j.

    Returns (sel, gap): sel is a length-k list of block ids, ascending, the
    diagonal j included, padded with -1; gap is, among the candidates the
    top-k choice ranks (b < j outside the always-kept window), S of the last
    one taken minus S of the first one left (inf when no choice is made).
    """
    forced = forced_blocks(j, window, dilation)
    if len(forced) > k - 1:
        raise ValueError("the always-kept window does not fit in top_k - 1 slots")
    cand_ids = [b for b in range(j) if b not in forced]
    free = k - 1 - len(forced)
    if len(cand_ids) <= free:
        chosen = cand_ids
        gap = math.inf
    else:
        cand = np.asarray([S_row[b] for b in cand_ids], dtype=np.float64)
        order = np.argsort(-cand, kind="stable")  # descending score, ties by lower b
        chosen = [cand_ids[int(n)] for n in order[:free]]
        gap = math.inf if free == 0 else float(cand[order[free - 1]] - cand[order[free]])
    sel = sorted(chosen + forced) + [j]
    sel = sel + [-1] * (k - len(sel))
    return sel, gap


def select_blocks(S: np.ndarray, rows: np.ndarray, prm: OracleParams):
    """Selection for every (row, group): sel [R, Hkv, k] int64, gap [R, Hkv]."""
    R = len(rows)
    sel = np.full((R, prm.hkv, prm.top_k), -1, dtype=np.int64)
    gap = np.full((R, prm.hkv), math.inf)
    for n, i in enumerate(rows):
        j = int(i) // prm.block
        for g in range(prm.hkv):
            s, gp = select_from_pooled(S[n, g, : j + 1], j, prm.top_k, prm.window, prm.dilation)
            sel[n, g] = s
            gap[n, g] = gp
    return sel, gap


# ---------------------------------------------------------------------------
# steps 4-9 for whole documents
# ---------------------------------------------------------------------------
def msa_reference(inputs: dict, prm: OracleParams, sel_override=None, arg_override=None,
                  with_grads: bool = True, row_chunk: int = 1024) -> dict:
    """Full forward + backward of one MSA training step, every row of every document.

    inputs: q [T,Hq,d], k/v [T,Hkv,d], q_p/k_p [T,Hkv,dp], dO [T,Hq,d], cu_seqlens.
    sel_override / arg_override ([T,Hkv,k] block ids / in-block argmax offsets)
    replace the oracle's own selection for steps 4-9 (used when comparing with
    another implementation whose choice differs only inside the tie band).
    """
    q, k, v = _f64(inputs["q"]), _f64(inputs["k"]), _f64(inputs["v"])
    q_p, k_p = _f64(inputs["q_p"]), _f64(inputs["k_p"])
    dO = _f64(inputs["dO"]) if with_grads else None
    T = q.shape[0]
    G, B, K = prm.group, prm.block, prm.top_k
    out = dict(
        sel_idx=np.full((T, prm.hkv, K), -1, dtype=np.int64),
        sel_score=np.zeros((T, prm.hkv, K)),
        sel_arg=np.zeros((T, prm.hkv, K), dtype=np.int64),
        own_sel_idx=np.full((T, prm.hkv, K), -1, dtype=np.int64),
        own_sel_arg=np.zeros((T, prm.hkv, K), dtype=np.int64),
        tie_gap=np.full((T, prm.hkv), math.inf),
        plse=np.zeros((T, prm.hkv)),
        pooled=[],
        o=np.zeros((T, prm.hq, prm.d)),
        lse=np.zeros((T, prm.hq)),
        mass=np.zeros((T, prm.hkv, K)),
        p=np.zeros((T, prm.hkv, K)),
        kl=np.zeros((T, prm.hkv)),
    )
    if with_grads:
        for name, shp in (("dq", q.shape), ("dk", k.shape), ("dv", v.shape), ("dq_p", q_p.shape),
                          ("dk_p", k_p.shape)):
            out[name] = np.zeros(shp)
    for (s0, s1) in doc_bounds(inputs["cu_seqlens"]):
        L = s1 - s0
        if L == 0:
            continue
        NB = (L + B - 1) // B
        rows = np.arange(L)
        S, A = pooled_proxy_scores(q_p[s0:s1], k_p[s0:s1], rows, prm)
        out["pooled"].append((s0, S))
        own_sel, gap = select_blocks(S, rows, prm)
        out["own_sel_idx"][s0:s1] = own_sel
        out["tie_gap"][s0:s1] = gap
        own_arg = np.zeros_like(own_sel)
        for g in range(prm.hkv):
            valid = own_sel[:, g, :] >= 0
            own_arg[:, g, :] = np.where(
                valid, A[rows[:, None], g, np.maximum(own_sel[:, g, :], 0)], 0)
        out["own_sel_arg"][s0:s1] = own_arg
        sel = own_sel if sel_override is None else _i64(sel_override)[s0:s1]
        arg = own_arg if arg_override is None else _i64(arg_override)[s0:s1]
        valid = sel >= 0
        sel_c = np.maximum(sel, 0)
        score = np.where(valid, S[rows[:, None, None], np.arange(prm.hkv)[None, :, None], sel_c],
                         NEG_INF)
        plse = _logsumexp(score, axis=2)  # [L, Hkv]
        out["sel_idx"][s0:s1] = sel
        out["sel_arg"][s0:s1] = np.where(valid, arg, 0)
        out["sel_score"][s0:s1] = np.where(valid, score, 0.0)
        out["plse"][s0:s1] = plse
        p = np.where(valid, np.exp(score - plse[:, :, None]), 0.0)
        out["p"][s0:s1] = p
        # block membership per (row, group): chosen[i, g, b]
        chosen = np.zeros((L, prm.hkv, NB), dtype=bool)
        for s in range(K):
            ok = valid[:, :, s]
            ii, gg = np.nonzero(ok)
            chosen[ii, gg, sel[ii, gg, s]] = True
        key_block = np.arange(L) // B
        mass = np.zeros((L, prm.hkv, K))
        for g in range(prm.hkv):
            kg, vg = k[s0:s1, g, :], v[s0:s1, g, :]
            for hh in range(G):
                h = g * G + hh
                for c0 in range(0, L, row_chunk):
                    c1 = min(L, c0 + row_chunk)
                    ri = np.arange(c0, c1)
                    M = (np.arange(L)[None, :] <= ri[:, None]) & chosen[c0:c1, g, :][:, key_block]
                    z = prm.softmax_scale * (q[s0 + c0:s0 + c1, h, :] @ kg.T)
                    z = np.where(M, z, NEG_INF)
                    lse = _logsumexp(z, axis=1)
                    P = np.where(M, np.exp(z - lse[:, None]), 0.0)
                    o = P @ vg
                    out["o"][s0 + c0:s0 + c1, h] = o
                    out["lse"][s0 + c0:s0 + c1, h] = lse
                    # per-block probability mass of this head
                    Ppad = np.zeros((c1 - c0, NB * B))
                    Ppad[:, :L] = P
                    blk_mass = Ppad.reshape(c1 - c0, NB, B).sum(axis=2)  # [r, NB]
                    mass[c0:c1, g, :] += np.where(
                        valid[c0:c1, g, :],
                        blk_mass[np.arange(c1 - c0)[:, None], sel_c[c0:c1, g, :]], 0.0) / G
                    if with_grads:
                        do = dO[s0 + c0:s0 + c1, h, :]
                        D = np.sum(do * o, axis=1)
                        dP = do @ vg.T
                        dS = P * (dP - D[:, None])
                        out["dq"][s0 + c0:s0 + c1, h] = prm.softmax_scale * (dS @ kg)
                        out["dk"][s0:s1, g] += prm.softmax_scale * (dS.T @ q[s0 + c0:s0 + c1, h, :])
                        out["dv"][s0:s1, g] += P.T @ do
        out["mass"][s0:s1] = mass
        with np.errstate(divide="ignore", invalid="ignore"):
            term = np.where(valid & (mass > 0), mass * (np.log(mass) - np.log(p)), 0.0)
        out["kl"][s0:s1] = term.sum(axis=2)
        if with_grads:
            gb = np.where(valid, prm.kl_weight * (p - mass), 0.0)  # [L, Hkv, K]
            key = sel_c * B + arg  # doc-local key index of each selected block's argmax
            for g in range(prm.hkv):
                for s in range(K):
                    ok = valid[:, g, s]
                    ii = np.nonzero(ok)[0]
                    kk = key[ii, g, s]
                    out["dq_p"][s0 + ii, g] += prm.proxy_scale * gb[ii, g, s][:, None] * k_p[s0 + kk, g]
                    np.add.at(out["dk_p"][:, g], s0 + kk,
                              prm.proxy_scale * gb[ii, g, s][:, None] * q_p[s0 + ii, g])
    out["kl_loss"] = prm.kl_weight * float(out["kl"].sum())
    return out


# ---------------------------------------------------------------------------
# the same steps for one query token (sampled rows of long sequences)
# ---------------------------------------------------------------------------
def row_reference(inputs: dict, prm: OracleParams, t: int, sel_override=None, arg_override=None,
                  contributions: bool = False, groups=None) -> dict:
    """Forward + backward quantities of one token t (all heads, all groups).

    Row-local outputs: sel (own selection), gap, sel_score, plse, o, lse, mass,
    p, kl, dq, dq_p.  With contributions=True also the row's additive
    contributions to dk / dv (per group: key indices and [n, d] rows) and to
    dk_p.  inputs may be torch tensors (bf16) or numpy arrays; only the rows
    that token t can see are upcast.  `groups` restricts the work to some KV
    groups (the others' entries stay zero).
    """
    cu = _i64(inputs["cu_seqlens"])
    doc = int(np.searchsorted(cu, t, side="right") - 1)
    s0 = int(cu[doc])
    i = t - s0
    B, K, G = prm.block, prm.top_k, prm.group
    j = i // B
    q_t = _f64(inputs["q"][t])  # [Hq, d]
    do_t = _f64(inputs["dO"][t])
    qp_t = _f64(inputs["q_p"][t])  # [Hkv, dp]
    kp = _f64(inputs["k_p"][s0:t + 1])  # [i+1, Hkv, dp] (a view when k_p is fp64 numpy)
    res = dict(sel=np.full((prm.hkv, K), -1, dtype=np.int64), gap=np.full(prm.hkv, math.inf),
               sel_score=np.zeros((prm.hkv, K)), sel_arg=np.zeros((prm.hkv, K), dtype=np.int64),
               own_arg=np.zeros((prm.hkv, K), dtype=np.int64),
               plse=np.zeros(prm.hkv), o=np.zeros((prm.hq, prm.d)), lse=np.zeros(prm.hq),
               mass=np.zeros((prm.hkv, K)), p=np.zeros((prm.hkv, K)), kl=np.zeros(prm.hkv),
               dq=np.zeros((prm.hq, prm.d)), dq_p=np.zeros((prm.hkv, prm.dp)),
               pooled=np.full((prm.hkv, j + 1), NEG_INF), contrib=[])
    for g in (range(prm.hkv) if groups is None else groups):
        s = prm.proxy_scale * (kp[:, g, :] @ qp_t[g])  # keys 0..i
        spad = np.full((j + 1) * B, NEG_INF)
        spad[: i + 1] = s
        blocks = spad.reshape(j + 1, B)
        S = blocks.max(axis=1)
        A = blocks.argmax(axis=1)
        res["pooled"][g] = S
        own, gap = select_from_pooled(S, j, K, prm.window, prm.dilation)
        res["gap"][g] = gap
        own_arr = np.asarray(own)
        res["own_arg"][g] = np.where(own_arr >= 0, A[np.maximum(own_arr, 0)], 0)
        sel = own_arr if sel_override is None else _i64(sel_override)[g]
        res["sel"][g] = own_arr
        valid = sel >= 0
        arg = (np.where(valid, A[np.maximum(sel, 0)], 0) if arg_override is None
               else _i64(arg_override)[g])
        score = np.where(valid, S[np.maximum(sel, 0)], NEG_INF)
        plse = _logsumexp(score, axis=0)
        p = np.where(valid, np.exp(score - plse), 0.0)
        res["sel_score"][g] = np.where(valid, score, 0.0)
        res["sel_arg"][g] = arg
        res["plse"][g] = plse
        res["p"][g] = p
        # keys of the selected blocks, causal (doc-local indices)
        keys = np.concatenate([np.arange(b * B, min((b + 1) * B, i + 1)) for b in sel[valid]])
        slot_of_key = np.concatenate([np.full(min((b + 1) * B, i + 1) - b * B, n)
                                      for n, b in enumerate(sel[valid])])
        kg = _f64(inputs["k"][s0 + keys, g])  # [n, d]
        vg = _f64(inputs["v"][s0 + keys, g])
        qh = q_t[g * G:(g + 1) * G]  # [G, d]
        z = prm.softmax_scale * (qh @ kg.T)  # [G, n]
        lse = _logsumexp(z, axis=1)
        P = np.exp(z - lse[:, None])
        o = P @ vg
        res["o"][g * G:(g + 1) * G] = o
        res["lse"][g * G:(g + 1) * G] = lse
        nvalid = int(valid.sum())
        mass = np.zeros(K)
        for n in range(nvalid):
            mass[n] = P[:, slot_of_key == n].sum() / G
        res["mass"][g] = mass
        with np.errstate(divide="ignore", invalid="ignore"):
            term = np.where(valid & (mass > 0), mass * (np.log(mass) - np.log(p)), 0.0)
        res["kl"][g] = term.sum()
        doh = do_t[g * G:(g + 1) * G]
        D = np.sum(doh * o, axis=1)
        dP = doh @ vg.T
        dS = P * (dP - D[:, None])
        res["dq"][g * G:(g + 1) * G] = prm.softmax_scale * (dS @ kg)
        gb = np.where(valid, prm.kl_weight * (p - mass), 0.0)
        akey = np.maximum(sel, 0) * B + arg
        kp_a = kp[akey[valid], g, :]  # [nvalid, dp]
        res["dq_p"][g] = prm.proxy_scale * (gb[valid][:, None] * kp_a).sum(axis=0)
        if contributions:
            res["contrib"].append(dict(
                g=g, keys=s0 + keys,
                dk=prm.softmax_scale * (dS.T @ qh),  # [n, d]
                dv=P.T @ doh,
                dkp_keys=s0 + akey[valid],
                dkp=prm.proxy_scale * gb[valid][:, None] * qp_t[g][None, :]))
    return res


def mask_pair_count(cu_seqlens, prm: OracleParams) -> int:
    """Number of (query head, key) pairs inside the selection mask, counted by
    enumerating rows: min(j, k-1) full off-diagonal blocks plus r+1 diagonal keys."""
    total = 0
    for (s0, s1) in doc_bounds(cu_seqlens):
        for i in range(s1 - s0):
            j, r = divmod(i, prm.block)
            total += min(j, prm.top_k - 1) * prm.block + r + 1
    return total * prm.hq


def effective_flops(cu_seqlens, prm: OracleParams) -> float:
    """Selected-block FLOPs of one fwd+bwd: 4d (fwd) + 10d (bwd) per masked pair."""
    return 14.0 * prm.d * mask_pair_count(cu_seqlens, prm)
