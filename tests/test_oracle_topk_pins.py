"""Pins for the oracle's top-k key selection, independent of the oracle's code.

The selection is the step that consumes the logits: the sparse-attention call
on the "FlashMLA" page takes ``indices`` of shape (batch, seq_len_q, topk)
with invalid entries set to -1.  The oracle's reading (largest values first by
IEEE-754 totalOrder, equal values to the smaller key, output in ascending key
order, -1 padding) is pinned here by hand-derived cases, by numpy's lexsort
(a library routine) on numeric order, by the special values where totalOrder
and numeric order part ways, and by invariants that any correct selection
satisfies.
"""
import numpy as np
import pytest


def f32(values):
    return np.asarray(values, dtype=np.float32)


def full_range(L):
    R, n = L.shape
    return np.zeros(R, np.int32), np.full(R, n, np.int32)


# ------------------------------------------------------------ hand-derived
def test_hand_example(oracle_mod):
    # values 3, 1, 2, 5 at keys 0..3: the two largest are 5 (key 3) and 3 (key 0)
    L = f32([[3.0, 1.0, 2.0, 5.0]])
    ks, ke = full_range(L)
    assert oracle_mod.topk_indices(L, ks, ke, topk=2).tolist() == [[0, 3]]
    # the three largest add 2 (key 2)
    assert oracle_mod.topk_indices(L, ks, ke, topk=3).tolist() == [[0, 2, 3]]
    # more slots than keys: every key, then -1
    assert oracle_mod.topk_indices(L, ks, ke, topk=6).tolist() == [[0, 1, 2, 3, -1, -1]]


def test_ties_go_to_smaller_key(oracle_mod):
    L = f32([[1.0, 1.0, 1.0, 1.0], [0.5, 2.0, 0.5, 0.5]])
    ks, ke = full_range(L)
    assert oracle_mod.topk_indices(L, ks, ke, topk=2).tolist() == [[0, 1], [0, 1]]
    assert oracle_mod.topk_indices(L, ks, ke, topk=3).tolist() == [[0, 1, 2], [0, 1, 2]]


def test_range_limits_candidates(oracle_mod):
    # keys 1 and 2 only: values 1 and 2, although key 3 holds the row's maximum
    L = f32([[3.0, 1.0, 2.0, 5.0]])
    got = oracle_mod.topk_indices(L, np.array([1], np.int32), np.array([3], np.int32), topk=3)
    assert got.tolist() == [[1, 2, -1]]
    # empty and inverted ranges select nothing
    for s, e in [(2, 2), (3, 1), (9, 12)]:
        got = oracle_mod.topk_indices(L, np.array([s], np.int32), np.array([e], np.int32), topk=2)
        assert got.tolist() == [[-1, -1]]


def test_total_order_special_values(oracle_mod):
    nan = np.float32(np.nan)
    neg_nan = np.frombuffer(np.uint32(0xFFC00000).tobytes(), np.float32)[0]
    cases = [
        ([-0.0, 0.0], 1, [1]),                   # +0 ranks above -0
        ([0.0, -0.0], 1, [0]),
        ([np.inf, nan], 1, [1]),                 # +NaN above +inf
        ([-np.inf, neg_nan], 1, [0]),            # -NaN below -inf
        ([-np.inf, -1e30, -np.inf], 2, [0, 1]),  # -inf is still a value
    ]
    for vals, k, want in cases:
        L = f32([vals])
        ks, ke = full_range(L)
        assert oracle_mod.topk_indices(L, ks, ke, topk=k).tolist() == [want], vals


# --------------------------------------------------- library routine (lexsort)
def lexsort_topk(row, lo, hi, k):
    keys = np.arange(lo, hi)
    vals = row[lo:hi].astype(np.float64)
    order = np.lexsort((keys, -vals))    # by value descending, then key ascending
    chosen = np.sort(keys[order[:k]])
    return np.concatenate([chosen, np.full(k - len(chosen), -1)]).astype(np.int32)


@pytest.mark.parametrize("seed,levels,k", [(1, 0, 5), (2, 4, 7), (3, 16, 40), (4, 1000, 1), (5, 3, 200)])
def test_matches_lexsort(oracle_mod, seed, levels, k):
    rng = np.random.default_rng(seed)
    R, n = 24, 150
    if levels:   # few distinct values: many ties at the threshold
        L = rng.integers(-levels, levels + 1, size=(R, n)).astype(np.float32) / 4
    else:
        L = rng.standard_normal((R, n)).astype(np.float32)
    L[rng.random((R, n)) < 0.05] = -np.inf
    ks = rng.integers(-5, n, size=R).astype(np.int32)
    ke = (ks + rng.integers(-3, n, size=R)).astype(np.int32)
    got = oracle_mod.topk_indices(L, ks, ke, topk=k)
    for i in range(R):
        lo, hi = max(int(ks[i]), 0), min(int(ke[i]), n)
        want = lexsort_topk(L[i], lo, max(hi, lo), k)
        assert np.array_equal(got[i], want), i


# ----------------------------------------------------------------- invariants
def test_selection_invariants(oracle_mod):
    rng = np.random.default_rng(11)
    R, n, k = 40, 300, 64
    L = (rng.integers(-20, 21, size=(R, n)) / 8).astype(np.float32)
    ks = rng.integers(0, 80, size=R).astype(np.int32)
    ke = (ks + rng.integers(0, 260, size=R)).astype(np.int32)
    got = oracle_mod.topk_indices(L, ks, ke, topk=k)
    for i in range(R):
        lo, hi = int(ks[i]), min(int(ke[i]), n)
        sel = got[i][got[i] >= 0]
        assert len(sel) == min(k, hi - lo)
        assert np.all(np.diff(sel) > 0) and np.all(got[i][len(sel):] == -1)
        assert np.all((sel >= lo) & (sel < hi))
        rest = np.setdiff1d(np.arange(lo, hi), sel)
        if len(rest):
            thr = L[i, sel].min()
            assert L[i, rest].max() <= thr
            # at the threshold value the smaller keys were taken
            tied_taken = sel[L[i, sel] == thr]
            tied_left = rest[L[i, rest] == thr]
            if len(tied_left):
                assert tied_taken.max() < tied_left.min()


def test_compressed_is_shifted_uncompressed(oracle_mod):
    rng = np.random.default_rng(12)
    R, n, ldo, k = 16, 200, 90, 20
    L = rng.standard_normal((R, n)).astype(np.float32)
    ks = rng.integers(0, 150, size=R).astype(np.int32)
    ke = (ks + rng.integers(0, 120, size=R)).astype(np.int32)
    C = np.full((R, ldo), np.nan, np.float32)
    for i in range(R):
        lo, hi = int(ks[i]), min(int(ke[i]), n, int(ks[i]) + ldo)
        C[i, :hi - lo] = L[i, lo:hi]
    got = oracle_mod.topk_indices(C, ks, ke, topk=k, n_cols=n, compressed=True)
    ke_cut = np.minimum(np.minimum(ke, n), ks + ldo).astype(np.int32)
    want = oracle_mod.topk_indices(L, ks, ke_cut, topk=k)
    assert np.array_equal(got, want)


def test_paged_ranges_follow_decode_rows(oracle_mod):
    # row r = b * next_n + t scores keys [0, ctx_b - next_n + t + 1)
    ctx = np.array([0, 1, 5, 9], np.int32)
    next_n = 3
    ks, ke = oracle_mod.paged_ranges(ctx, next_n)
    want = []
    for b in range(len(ctx)):
        for t in range(next_n):
            want.append(max(int(ctx[b]) - next_n + t + 1, 0))
    assert ks.tolist() == [0] * len(want) and ke.tolist() == want
    rng = np.random.default_rng(13)
    L = rng.standard_normal((len(want), 12)).astype(np.float32)
    got = oracle_mod.paged_topk_indices(L, ctx, next_n=next_n, topk=4)
    assert np.array_equal(got, oracle_mod.topk_indices(L, ks, ke, topk=4))


def test_rows_slice_matches_whole(oracle_mod):
    rng = np.random.default_rng(14)
    L = rng.standard_normal((10, 50)).astype(np.float32)
    ks, ke = full_range(L)
    whole = oracle_mod.topk_indices(L, ks, ke, topk=7)
    assert np.array_equal(oracle_mod.topk_indices(L, ks, ke, topk=7, rows=(3, 8)), whole[3:8])


def test_invalid_arguments(oracle_mod):
    L = f32([[1.0, 2.0]])
    ks, ke = full_range(L)
    with pytest.raises(ValueError):
        oracle_mod.topk_indices(L, ks, ke, topk=0)
    with pytest.raises(ValueError):
        oracle_mod.topk_indices(L, ks, ke, topk=1, n_cols=3)   # uncompressed row wider than ldo
