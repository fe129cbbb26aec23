"""Shared comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (floating point, bf16 inputs, fp32 accumulation on the GPU):
cosine similarity >= 0.9995 and max |gpu - oracle| <= 2e-2 for O, dQ, dK, dV,
dq_p, dk_p; the KL loss to 1e-3 relative.  Integer outputs (block indices,
argmax offsets, regroup lists) are compared exactly, except where the oracle's
(k-1)-th and k-th best pooled scores lie within 1e-3 of each other: there the
differing blocks must all sit inside that tie band.
"""
from __future__ import annotations

import numpy as np

COS_MIN = 0.9995
ABS_MAX = 2e-2
TIE_BAND = 1e-3
KL_RTOL = 1e-3


def cos(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb + 1e-300))


def assert_close(name, gpu, ref, cos_min=COS_MIN, abs_max=ABS_MAX):
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite GPU values"
    e = float(np.abs(g - r).max()) if g.size else 0.0
    if g.size == 0 or float(np.abs(r).max()) < 1e-9:
        # an identically-zero quantity (e.g. the proxy gradient when every row
        # keeps a single block): the cosine is undefined, only the abs bound applies
        assert e <= abs_max, f"{name}: max-abs {e:.3e} (<= {abs_max}) on a zero reference"
        return 1.0, e
    c = cos(g, r)
    assert c >= cos_min and e <= abs_max, f"{name}: cos {c:.6f} (>= {cos_min}), max-abs {e:.3e} (<= {abs_max})"
    return c, e


def check_selection_row(gpu_sel, own_sel, pooled, j, k, window=0, dilation=1):
    """One (row, group): GPU and oracle block lists must agree, or differ only in
    blocks whose oracle pooled score is within TIE_BAND of the selection boundary.
    With a block pattern (window, dilation) the always-kept blocks must be in
    the GPU's list and are not ranked.  Returns True when the row is an excused tie."""
    gpu_sel = [int(x) for x in gpu_sel]
    own_sel = [int(x) for x in own_sel]
    n_off = min(j, k - 1)
    kept = {j - dilation * u for u in range(1, window + 1) if j - dilation * u >= 0}
    assert kept <= set(gpu_sel[:n_off]), (gpu_sel, sorted(kept))
    if gpu_sel == own_sel:
        return False
    # structure: ascending, diagonal last, -1 padding
    assert gpu_sel[n_off] == j and all(x == -1 for x in gpu_sel[n_off + 1:]), gpu_sel
    assert gpu_sel[:n_off] == sorted(set(gpu_sel[:n_off])), gpu_sel
    free = n_off - len(kept)  # slots the ranking fills
    ranked = np.asarray([b for b in range(j) if b not in kept])
    assert free >= 1 and len(ranked) > free, f"no choice to tie on: {gpu_sel} vs {own_sel}"
    cand = np.asarray(pooled[:j], np.float64)
    srt = np.sort(cand[ranked])[::-1]
    lo = srt[free]        # best excluded
    hi = srt[free - 1]    # worst included
    assert hi - lo < TIE_BAND, f"selection differs outside the tie band: {gpu_sel} vs {own_sel}"
    diff = set(gpu_sel[:n_off]) ^ set(own_sel[:n_off])
    for b in diff:
        assert b not in kept and lo - TIE_BAND <= cand[b] <= hi + TIE_BAND, (b, cand[b], lo, hi)
    return True


# The kernel compares fp32 pooled scores (bf16 products summed in fp32), the
# oracle fp64 ones; they differ by well under 1e-5 (sel_score agrees to 1e-3
# by assertion and to ~1e-6 in practice).  A row whose fp64 gap lies within
# this margin of the band edge may fall on either side of it.
TIE_MARGIN = 1e-4


def check_tie_flags(gpu_tie, gap, band=TIE_BAND, margin=TIE_MARGIN):
    """The GPU's tie flag [rows, Hkv] against the oracle's selection gap (S of
    the last ranked block taken minus S of the first left; inf when the row
    makes no choice): every flag must equal (gap < band), except rows whose gap
    lies within `margin` of the band edge.  Returns the number of such excused
    rows (flags that differ from the fp64 reading)."""
    t = np.asarray(gpu_tie).astype(np.int64)
    gap = np.asarray(gap, np.float64)
    assert t.shape == gap.shape, (t.shape, gap.shape)
    assert np.isin(t, (0, 1)).all(), "tie flag holds a value other than 0 or 1"
    want = (gap < band).astype(np.int64)
    near = np.abs(gap - band) <= margin
    bad = (t != want) & ~near
    if bad.any():
        idx = tuple(int(x[0]) for x in np.nonzero(bad))
        raise AssertionError(f"tie flag differs from (gap < {band}) at {int(bad.sum())} "
                             f"(row, group) pairs; first {idx}: gpu {t[idx]}, gap {gap[idx]:.6g}")
    return int(((t != want) & near).sum())


def check_argmax_row(gpu_sel, gpu_arg, own_sel, own_arg, pooled, score_of):
    """Argmax offsets of one (row, group).  Where the GPU's block list equals the
    oracle's and an offset equals the oracle's (lowest key attaining the max),
    nothing more is checked; otherwise the fp64 score of the GPU's key,
    score_of(block, offset), must lie within TIE_BAND below the block's fp64
    maximum pooled[block] (an argmax tie).  Returns the number of offsets that
    differ from the oracle's."""
    same_list = [int(x) for x in gpu_sel] == [int(x) for x in own_sel]
    n = 0
    for s, b in enumerate(gpu_sel):
        b = int(b)
        if b < 0:
            continue
        a = int(gpu_arg[s])
        if same_list and a == int(own_arg[s]):
            continue
        sc = float(score_of(b, a))
        assert pooled[b] - TIE_BAND < sc <= pooled[b] + 1e-9, (s, b, a, sc, pooled[b])
        n += 1
    return n
