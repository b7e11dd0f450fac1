"""Top-k key selection on the GPU (through the C ABI) against the CPU oracle.

The selection is unique (larger value by totalOrder first, ties to the smaller
key, output in ascending key order, -1 padding), so every case compares the
whole index matrix bit for bit with the oracle run on the same logits bytes.
Cases cover ragged, empty, inverted and clipped ranges, rows shorter than,
equal to and just longer than topk, many exact ties (including rows whose
threshold bin overflows shared memory), special values, unaligned row starts,
the compressed layout, 65536-key rows, the full 2048 x 32768 workload the
benchmark times, and the logits -> top-k pipeline for dense and paged calls.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU suite needs a CUDA device"
    from fp8_mqa_indexer_gb300 import build
    build.build()
    oracle.build()
    return torch.device("cuda:0")


def oracle_topk(L, ks, ke, topk, n_cols, compressed=False):
    """Oracle over all rows, spread over host threads (rows are independent)."""
    L = L.detach().cpu().numpy() if hasattr(L, "detach") else L
    rows = L.shape[0]
    step = max(1, rows // 64)
    spans = [(a, min(rows, a + step)) for a in range(0, rows, step)]
    res = oracle.run_rows_parallel(
        lambda sp: oracle.topk_indices(L, ks, ke, topk=topk, n_cols=n_cols, compressed=compressed,
                                       rows=sp), spans)
    return np.concatenate([res[sp] for sp in spans]) if spans else np.zeros((0, topk), np.int32)


def gpu_topk(L, ks, ke, topk, n_cols, dev, compressed=False):
    out = mqa.mqa_topk_indices(L, ks.to(dev), ke.to(dev), topk, S_kv=n_cols, compressed=compressed)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check(case, dev, *, offset=0):
    """GPU against oracle; ``offset`` > 0 shifts every row start off a 16-byte boundary."""
    L = case.logits
    if offset:
        big = torch.full((case.rows, case.ldo + offset), float("nan"))
        big[:, offset:] = L
        Ld = big.to(dev)[:, offset:]
    else:
        Ld = L.to(dev)
    got = gpu_topk(Ld, case.k_start, case.k_end, case.topk, case.n_cols, dev, case.compressed)
    want = oracle_topk(L, case.k_start, case.k_end, case.topk, case.n_cols, case.compressed)
    if not np.array_equal(got, want):
        r = int(np.nonzero((got != want).any(axis=1))[0][0])
        c = int(np.nonzero(got[r] != want[r])[0][0])
        raise AssertionError(f"{case.name}: {int((got != want).any(axis=1).sum())} rows differ; first "
                             f"row {r} at slot {c}: gpu {got[r, c]} oracle {want[r, c]}")


# ------------------------------------------------------------ small cases
def ragged_ranges(n_cols, topk):
    starts = [0, 0, 5, 0, 0, 0, 3, -7, 10, n_cols - 1, n_cols, 50, 0]
    ends = [0, 1, 5 + topk - 1, topk, topk + 1, n_cols, n_cols + 9, 40, 3, n_cols, n_cols + 5,
            50 + 3 * topk, n_cols - 1]
    return starts, ends


@pytest.mark.parametrize("n_cols,topk,levels", [
    (300, 7, 0), (300, 7, 2), (5000, 64, 0), (5000, 64, 1), (20000, 2048, 0), (20000, 2048, 2),
    (20000, 1, 0), (4099, 512, 8)])
def test_ragged_rows(dev, n_cols, topk, levels):
    ks, ke = ragged_ranges(n_cols, topk)
    case = wl.topk_case(len(ks), n_cols, topk, seed=700 + n_cols + topk + levels, ranges="custom",
                        levels=levels, k_start=ks, k_end=ke, name=f"ragged n={n_cols} k={topk}")
    check(case, dev)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_rows(dev, offset):
    case = wl.topk_case(24, 3001, 100, seed=710 + offset, ranges="causal_tail", ldo=3003,
                        name=f"unaligned +{offset}")
    check(case, dev, offset=offset)


def test_many_rows_and_ties(dev):
    # more rows than the grid holds at once, coarse values: many exact ties
    case = wl.topk_case(700, 6000, 300, seed=720, ranges="causal_tail", levels=4, name="700 rows")
    check(case, dev)


def test_threshold_bin_overflow(dev):
    # all values equal, or two levels only: the threshold bin holds far more
    # elements than shared memory, so the selection re-reads the row
    n = 30000
    L = torch.full((4, n), 0.25)
    L[1] = torch.where(torch.arange(n) % 3 == 0, 1.0, 0.5)
    L[2, ::2] = -0.0
    L[2, 1::2] = 0.0
    L[3] = torch.linspace(-1, 1, n)
    case = wl.TopkCase("overflow", L, torch.zeros(4, dtype=torch.int32),
                       torch.full((4,), n, dtype=torch.int32), n, 12000)
    check(case, dev)


def test_special_values(dev):
    g = torch.Generator().manual_seed(730)
    n = 9000
    L = torch.randn((8, n), generator=g)
    pick = torch.rand((8, n), generator=g)
    L[pick < 0.05] = float("inf")
    L[(pick >= 0.05) & (pick < 0.08)] = float("-inf")
    L[(pick >= 0.08) & (pick < 0.10)] = float("nan")
    neg_nan = torch.tensor([0xFFC00000], dtype=torch.int64).to(torch.int32).view(torch.float32)[0]
    L[(pick >= 0.10) & (pick < 0.12)] = neg_nan
    L[(pick >= 0.12) & (pick < 0.2)] = -0.0
    L[(pick >= 0.2) & (pick < 0.3)] = 0.0
    case = wl.TopkCase("special", L, torch.zeros(8, dtype=torch.int32),
                       torch.full((8,), n, dtype=torch.int32), n, 1000)
    check(case, dev)


def test_compressed_layout(dev):
    n_cols, ldo, rows = 5000, 1500, 40
    g = torch.Generator().manual_seed(740)
    ks = torch.randint(-10, n_cols, (rows,), generator=g, dtype=torch.int32)
    ke = ks + torch.randint(-5, 2500, (rows,), generator=g, dtype=torch.int32)
    case = wl.topk_case(rows, n_cols, 300, seed=741, ranges="custom", k_start=ks, k_end=ke,
                        ldo=ldo, name="compressed")
    case.compressed = True   # columns hold keys k_start + c; the range is cut at ldo
    check(case, dev)


def test_long_rows(dev):
    case = wl.topk_case(6, 65536, 2048, seed=750, ranges="full", name="65536 keys")
    check(case, dev)
    case = wl.topk_case(3, 65536, 2048, seed=751, ranges="full", levels=1, name="65536 keys, ties")
    check(case, dev)


@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_one_pass_rows_unaligned(dev, offset):
    """Rows long enough for the sampled one-pass selection, starting and ending
    at every alignment (row starts shifted off 16 bytes, ldo odd, range ends
    at arbitrary columns), uncompressed and compressed."""
    n_cols, rows = 20001, 12
    g = torch.Generator().manual_seed(770 + offset)
    ks = torch.randint(0, 40, (rows,), generator=g, dtype=torch.int32)
    ke = n_cols - torch.randint(0, 40, (rows,), generator=g, dtype=torch.int32)
    case = wl.topk_case(rows, n_cols, 1000, seed=771 + offset, ranges="custom", k_start=ks,
                        k_end=ke, ldo=n_cols + 2, name=f"one-pass +{offset}")
    check(case, dev, offset=offset)
    case = wl.topk_case(rows, n_cols, 1000, seed=775 + offset, ranges="custom", k_start=ks,
                        k_end=ke, ldo=n_cols + 2, name=f"one-pass compressed +{offset}")
    case.compressed = True
    check(case, dev, offset=offset)


def test_rows_around_the_one_pass_limits(dev):
    """Row lengths on both sides of the shortest row that takes the sampled
    one-pass selection at k = 2048 (8192 keys), just above k, and long rows,
    in one call."""
    lens = [8190, 8191, 8192, 8193, 2049, 34809, 40000, 2048]
    n_cols = max(lens) + 5
    ks = torch.tensor([1, 2, 3, 0, 4, 1, 0, 7], dtype=torch.int32)
    ke = ks + torch.tensor(lens, dtype=torch.int32)
    case = wl.topk_case(len(lens), n_cols, 2048, seed=780, ranges="custom", k_start=ks, k_end=ke,
                        name="one-pass limits")
    check(case, dev)
    check(case, dev, offset=1)


def test_deterministic(dev):
    case = wl.topk_case(64, 20000, 2048, seed=760, ranges="causal_tail", levels=3)
    Ld = case.logits.to(dev)
    a = gpu_topk(Ld, case.k_start, case.k_end, case.topk, case.n_cols, dev)
    b = gpu_topk(Ld, case.k_start, case.k_end, case.topk, case.n_cols, dev)
    assert np.array_equal(a, b)


# ------------------------------------------------------- full-size workload
def test_full_workload(dev):
    case = wl.topk_config("topk_2k_32k_k2048")
    check(case, dev)


# --------------------------------------------------------------- pipelines
def test_dense_logits_then_topk(dev):
    """mqa_logits on the 2048 x 32768 workload, then top-2048 on its output;
    the oracle selects from the same logits bytes."""
    case = wl.dense_config("dense_2k_32k_h64_d128")
    q, kv = case.q.to(dev), case.kv.to(dev)
    s, w = case.kv_scale.to(dev), case.weights.to(dev)
    ks, ke = case.k_start.to(dev), case.k_end.to(dev)
    logits = mqa.mqa_logits(q, kv, s, w, ks, ke)
    idx = mqa.mqa_topk_indices(logits, ks, ke, 2048)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    want = oracle_topk(logits.cpu(), case.k_start, case.k_end, 2048, case.S_kv)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_paged_logits_then_topk(dev):
    B, next_n = 6, 2
    ctx = [1, 0, 129, 700, 64, 3000]
    case = wl.paged_case(B, next_n, 64, 128, seed=770, ctx_lo=0, ctx_hi=3072, block_kv=64,
                         num_blocks=200, context_lens=ctx)
    d = dict(q=case.q.to(dev), kvc=case.kv_cache.to(dev), sc=case.kv_scales.to(dev),
             w=case.weights.to(dev), cl=case.context_lens.to(dev), bt=case.block_table.to(dev))
    meta = mqa.paged_mqa_logits_metadata(d["cl"], next_n=next_n, block_kv=case.block_kv)
    logits = mqa.paged_mqa_logits(d["q"], d["kvc"], d["sc"], d["w"], d["cl"], d["bt"], meta,
                                  next_n=next_n)
    for topk in (1, 64, 700, 5000):
        idx = mqa.paged_mqa_topk_indices(logits, d["cl"], topk, next_n=next_n)
        torch.cuda.synchronize()
        want = oracle.paged_topk_indices(logits.cpu().numpy(), case.context_lens, next_n=next_n,
                                         topk=topk)
        assert np.array_equal(idx.cpu().numpy(), want), topk
    assert mqa.device_status() == 0


def test_row_split_matches_whole(dev):
    """Row slabs selected by separate calls (views into the same logits, as
    one rank per GPU would run them) give the whole call's rows bit for bit."""
    from fp8_mqa_indexer_gb300 import sharding
    case = wl.topk_case(301, 20000, 2048, seed=780, ranges="causal_tail", levels=2)
    Ld, ks, ke = case.logits.to(dev), case.k_start.to(dev), case.k_end.to(dev)
    whole = mqa.mqa_topk_indices(Ld, ks, ke, case.topk, S_kv=case.n_cols)
    parts = []
    for rank in range(3):
        v, _ = sharding.topk_row_shard(Ld, ks, ke, rank, 3)
        parts.append(mqa.mqa_topk_indices(v["logits"], v["k_start"], v["k_end"], case.topk,
                                          S_kv=case.n_cols))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts), whole)
