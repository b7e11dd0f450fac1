"""CPU check of the fused logits + top-k call's selection argument (no GPU).

The fused call writes, for each row, every logit of a tail of its range and,
of the rest, only the logits not below T, the tail's topk-th largest logit;
then it selects the topk largest among what it wrote.  The claim is that this
equals the top-k of the whole row (at least topk logits are >= T, and every
one of them is written).  This test restates the split and the candidate rule
in numpy and checks the claim against the oracle's top-k on rows with ties,
signed zeros, infinities and NaNs, at lengths around the split's thresholds.
"""
import math

import numpy as np
import pytest

import oracle


def order_key(v: np.ndarray) -> np.ndarray:
    """Unsigned keys whose order is the IEEE-754 totalOrder of the fp32 values."""
    u = v.astype(np.float32).view(np.uint32)
    flip = np.where(u >> 31 == 1, np.uint32(0xFFFFFFFF), np.uint32(0x80000000))
    return u ^ flip


def fused_topk_row(row: np.ndarray, lo: int, hi: int, k: int) -> np.ndarray:
    """The fused call's selection for one row, restated: candidates, then the
    top-k of the candidates (larger totalOrder first, ties to the smaller
    key), in ascending key order, -1 padded."""
    n = hi - lo
    out = np.full(k, -1, np.int32)
    if n <= k:
        out[:n] = np.arange(lo, hi)
        return out
    length = max(2 * k, math.ceil(math.sqrt(n * k)))
    length = (length + 127) // 128 * 128
    s = max(lo, (hi - length) // 128 * 128)
    keys = order_key(row)
    cand = np.zeros(len(row), bool)
    if s > lo:
        tail = np.sort(keys[s:hi])[::-1]
        T = tail[k - 1]                               # the tail's topk-th largest key
        T_f = np.array([T ^ (0x80000000 if T >> 31 else 0xFFFFFFFF)], np.uint32).view(np.float32)[0]
        cand[s:hi] = keys[s:hi] >= T                  # tail: filtered by the exact key
        rest = row[lo:s]
        with np.errstate(invalid="ignore"):
            cand[lo:s] = ~(rest < T_f)                # rest: written unless below T
        assert cand.sum() >= k
    else:
        cand[lo:hi] = True
    idx = np.nonzero(cand)[0]
    order = np.lexsort((idx, -keys[idx].astype(np.int64)))
    taken = np.sort(idx[order[:k]])
    out[:k] = taken
    return out


def special_row(n: int, g: np.random.Generator, kind: str) -> np.ndarray:
    if kind == "normal":
        return g.standard_normal(n).astype(np.float32)
    if kind == "coarse":                              # many exact ties
        return (np.round(g.standard_normal(n) * 2) / 2).astype(np.float32)
    if kind == "zeros":                               # +0 and -0 only
        v = np.zeros(n, np.float32)
        v[g.random(n) < 0.5] = -0.0
        return v
    v = g.standard_normal(n).astype(np.float32)       # specials mixed in
    p = g.random(n)
    v[p < 0.03] = np.inf
    v[(p >= 0.03) & (p < 0.05)] = -np.inf
    v[(p >= 0.05) & (p < 0.06)] = np.nan
    v[(p >= 0.06) & (p < 0.07)] = -np.nan
    v[(p >= 0.07) & (p < 0.09)] = -0.0
    return v


@pytest.mark.parametrize("kind", ["normal", "coarse", "zeros", "special"])
@pytest.mark.parametrize("n,k", [(3000, 64), (4100, 1024), (2049, 1024), (2177, 1024),
                                 (5000, 1), (700, 300), (20000, 2048), (301, 300)])
def test_fused_selection_equals_row_topk(kind, n, k):
    g = np.random.default_rng(n * 7 + k + len(kind))
    width = n + 200
    rows = []
    ranges = [(0, n), (37, 37 + n), (200, n + 200), (5, 5 + min(n, k)), (90, 80)]
    for lo, hi in ranges:
        r = np.full(width, np.nan, np.float32)
        r[max(lo, 0):max(hi, lo)] = special_row(max(hi - lo, 0), g, kind)
        rows.append(r)
    L = np.stack(rows)
    ks = np.array([a for a, _ in ranges], np.int32)
    ke = np.array([b for _, b in ranges], np.int32)
    want = oracle.topk_indices(L, ks, ke, topk=k, n_cols=width)
    for i, (lo, hi) in enumerate(ranges):
        lo_c, hi_c = min(max(lo, 0), width), max(min(hi, width), min(max(lo, 0), width))
        got = fused_topk_row(L[i], lo_c, hi_c, k)
        assert np.array_equal(got, want[i]), (kind, n, k, i)
