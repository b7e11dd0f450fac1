"""Fused logits + top-k (``mqa_logits_topk``) on the GPU, through the C ABI.

The fused call never writes the logits.  Each case therefore computes them a
second time with ``mqa_logits`` (the same per-logit arithmetic, so the same
fp32 bytes) and checks the fused indices bit for bit against the oracle's
selection over those bytes and against ``mqa_topk_indices`` over them.  Small
cases are also checked against the oracle's own logits: every selected key
must be, within the oracle's error bound, at least as large as every key left
out.  Cases cover ragged, empty, inverted and clipped ranges, rows shorter
than, equal to and just longer than topk, rows whose tail holds the whole
range, exact ties, topk above the shared list, negative key scales, every
(H, D) instance, bf16 weights, a workspace full of garbage, replay from a CUDA
graph, and the 2048 x 32768 and 8192 x 65536 workloads.
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


def to_dev(case, dev):
    return dict(q=case.q.to(dev), kv=case.kv.to(dev), s=case.kv_scale.to(dev),
                w=case.weights.to(dev), ks=case.k_start.to(dev), ke=case.k_end.to(dev))


def fused(d, topk, workspace=None):
    idx = mqa.mqa_logits_topk(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], topk,
                              workspace=workspace)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    return idx.cpu().numpy()


def plain_logits(d):
    """The logits of the same inputs, written out (non-clean: positions
    outside a range are never read by the selection)."""
    S_q, S_kv = d["q"].shape[0], d["kv"].shape[0]
    L = torch.full((S_q, S_kv), float("nan"), device=d["q"].device)
    mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], L, clean=False)
    torch.cuda.synchronize()
    return L


def oracle_topk_rows(L, ks, ke, topk, n_cols, rows=None):
    L = L.cpu().numpy() if hasattr(L, "cpu") else L
    R = L.shape[0]
    rows = list(range(R)) if rows is None else list(rows)
    step = max(1, len(rows) // 64)
    spans = [rows[a:a + step] for a in range(0, len(rows), step)]

    def one(span):
        return np.concatenate([oracle.topk_indices(L, ks, ke, topk=topk, n_cols=n_cols,
                                                   rows=(r, r + 1)) for r in span])
    res = oracle.run_rows_parallel(lambda i: one(spans[i]), list(range(len(spans))))
    return np.concatenate([res[i] for i in range(len(spans))])


def check_against_written_logits(case, dev, topk, **kw):
    d = to_dev(case, dev)
    got = fused(d, topk, **kw)
    L = plain_logits(d)
    want = oracle_topk_rows(L, case.k_start, case.k_end, topk, case.S_kv)
    if not np.array_equal(got, want):
        r = int(np.nonzero((got != want).any(axis=1))[0][0])
        c = int(np.nonzero(got[r] != want[r])[0][0])
        raise AssertionError(f"{case.name} topk={topk}: {int((got != want).any(axis=1).sum())} rows "
                             f"differ; row {r} slot {c}: fused {got[r, c]} oracle {want[r, c]}")
    unfused = mqa.mqa_topk_indices(L, d["ks"], d["ke"], topk, S_kv=case.S_kv)
    torch.cuda.synchronize()
    assert np.array_equal(got, unfused.cpu().numpy())
    return got


def check_within_oracle_bound(case, got, topk):
    """The selection against the oracle's own logits (fp64, rounded once): a
    valid top-k within the oracle's per-logit error bound."""
    L, tol = oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                               case.k_end, clean=False, with_tol=True)
    n_cols = case.S_kv
    for i in range(L.shape[0]):
        lo = min(max(int(case.k_start[i]), 0), n_cols)
        hi = max(min(int(case.k_end[i]), n_cols), lo)
        n = hi - lo
        sel = got[i][got[i] >= 0]
        assert len(sel) == min(n, topk) and np.all(got[i][len(sel):] == -1)
        assert np.all(np.diff(sel) > 0) and (len(sel) == 0 or (sel[0] >= lo and sel[-1] < hi))
        if n <= topk:
            continue
        rest = np.setdiff1d(np.arange(lo, hi), sel)
        low_sel = np.min(L[i, sel].astype(np.float64) + tol[i, sel])
        high_rest = np.max(L[i, rest].astype(np.float64) - tol[i, rest])
        assert low_sel >= high_rest, (case.name, i, low_sel, high_rest)


def ragged(S_kv, topk):
    """Row ranges: empty, inverted, clipped, shorter than / equal to / just
    longer than topk, tails that hold the whole range, long rows, odd starts."""
    pre = max(2 * topk, 128)
    ks = [0, 5, 9, 0, 0, 0, -30, S_kv - 3, S_kv, 3, 1, 7, 0, 0, 33, 100, S_kv // 2, 0, 17, 64]
    ke = [0, 5, 2, topk, topk + 1, S_kv, 40, S_kv + 50, S_kv + 9, 3 + topk - 1, 1 + pre, 7 + pre + 1,
          pre + 129, S_kv - 1, S_kv, S_kv - 7, S_kv, 31, S_kv - 100, 64 + 3 * topk]
    return ks, ke


@pytest.mark.parametrize("S_kv,topk", [(3001, 1), (3001, 64), (3001, 300), (4100, 1024),
                                       (2000, 5000)])
def test_ragged_rows(dev, S_kv, topk):
    ks, ke = ragged(S_kv, topk)
    case = wl.dense_case(len(ks), S_kv, 64, 128, seed=900 + S_kv + topk, ranges="custom",
                         k_start=ks, k_end=ke, clean=False, name=f"ragged {S_kv}")
    got = check_against_written_logits(case, dev, topk)
    check_within_oracle_bound(case, got, topk)


def test_topk_above_the_shared_list(dev):
    # topk 5000 > the 4096-entry shared list: rows with a remainder take the
    # selection's full digit path over the candidates
    S_kv = 20000
    ks = [0, 0, 0, 100, 3, 0, 7000, 0, 0, 15000]
    ke = [S_kv, 19999, 12000, S_kv, 10007, 5001, S_kv, 4999, 0, S_kv]
    case = wl.dense_case(len(ks), S_kv, 64, 128, seed=990, ranges="custom", k_start=ks, k_end=ke,
                         clean=False, name="topk 5000")
    got = check_against_written_logits(case, dev, 5000)
    check_within_oracle_bound(case, got, 5000)


@pytest.mark.parametrize("H,D", [(8, 64), (32, 64), (64, 64), (8, 128), (32, 128)])
def test_every_instance(dev, H, D):
    case = wl.dense_case(70, 2500, H, D, seed=910 + H + D, ranges="causal_tail", clean=False,
                         name=f"H{H} D{D}")
    got = check_against_written_logits(case, dev, 200)
    check_within_oracle_bound(case, got, 200)


def test_query_blocks_span_many_tiles(dev):
    # 129 rows: several query blocks, a ragged last block, suffix ranges
    case = wl.dense_case(129, 9000, 64, 128, seed=920, ranges="suffix", clean=False, name="suffix")
    check_against_written_logits(case, dev, 512)


def test_exact_ties(dev):
    # zero weights: every logit is +0, so the selection is the smallest keys
    case = wl.dense_case(40, 3000, 64, 128, seed=930, ranges="causal_tail", clean=False,
                         name="ties")
    case.weights.zero_()
    got = check_against_written_logits(case, dev, 100)
    for i in range(40):
        n = max(int(case.k_end[i]), 0)
        assert np.array_equal(got[i][:min(n, 100)], np.arange(min(n, 100)))
    # rows longer than the shared list, all equal: every estimate fails and
    # the selection walks the candidates for each digit
    case = wl.dense_case(6, 9000, 64, 128, seed=932, ranges="full", clean=False, name="long ties")
    case.weights.zero_()
    got = check_against_written_logits(case, dev, 1000)
    assert np.array_equal(got, np.tile(np.arange(1000, dtype=np.int32), (6, 1)))
    # coarse inputs: many equal logits, not all
    case = wl.dense_case(40, 5000, 32, 64, seed=931, ranges="full", clamp=0.5, clean=False,
                         name="coarse")
    check_against_written_logits(case, dev, 700)


def test_negative_key_scales(dev):
    case = wl.dense_case(50, 4000, 64, 128, seed=940, ranges="causal_tail", clean=False,
                         name="negative scales")
    g = torch.Generator().manual_seed(941)
    flip = torch.rand(case.S_kv, generator=g) < 0.3
    case.kv_scale[flip] = -case.kv_scale[flip]
    case.kv_scale[::97] = 0.0
    got = check_against_written_logits(case, dev, 256)
    check_within_oracle_bound(case, got, 256)


def test_bf16_weights(dev):
    case = wl.dense_case(33, 3000, 64, 128, seed=950, ranges="causal_tail", clean=False,
                         name="bf16 weights")
    case.weights = case.weights.to(torch.bfloat16)
    d = to_dev(case, dev)
    got = fused(d, 128)
    L = plain_logits(d)
    want = oracle_topk_rows(L, case.k_start, case.k_end, 128, case.S_kv)
    assert np.array_equal(got, want)
    # and the same as fp32 weights holding the bf16 values
    d32 = dict(d, w=d["w"].float())
    assert np.array_equal(fused(d32, 128), got)


def test_garbage_workspace_and_reuse(dev):
    """Nothing is read from the workspace that the call did not write."""
    case = wl.dense_case(64, 6000, 64, 128, seed=960, ranges="causal_tail", clean=False,
                         name="workspace")
    d = to_dev(case, dev)
    ref = fused(d, 400)
    nbytes = mqa.mqa_logits_topk_workspace_size(64, 6000)
    for fill in (0xff, 0x00, 0x7f):
        ws = torch.full((nbytes,), fill, dtype=torch.uint8, device=dev)
        assert np.array_equal(fused(d, 400, ws), ref)
    g = torch.Generator(device=dev).manual_seed(961)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev, generator=g)
    assert np.array_equal(fused(d, 400, ws), ref)
    # the same workspace, a different problem, then the first again
    other = wl.dense_case(64, 6000, 64, 128, seed=962, ranges="suffix", clean=False, name="o")
    fused(to_dev(other, dev), 50, ws)
    assert np.array_equal(fused(d, 400, ws), ref)


def test_no_keys(dev):
    case = wl.dense_case(5, 0, 64, 128, seed=970, ranges="full", clean=False, name="no keys")
    d = to_dev(case, dev)
    got = fused(d, 8)
    assert np.all(got == -1)


def test_deterministic(dev):
    case = wl.dense_case(256, 20000, 64, 128, seed=980, ranges="causal_tail", clean=False,
                         name="repeat")
    d = to_dev(case, dev)
    first = fused(d, 2048)
    for _ in range(19):
        assert np.array_equal(fused(d, 2048), first)


@pytest.mark.parametrize("name", ["dense_2k_32k_h64_d128", "dense_8k_64k_h64_d128"])
def test_full_workloads_equal_the_unfused_pipeline(dev, name):
    """At the benchmark sizes: the fused indices equal mqa_topk_indices over
    the mqa_logits output on every row, and the oracle agrees on sampled rows."""
    case = wl.dense_config(name)
    d = to_dev(case, dev)
    got = fused(d, 2048)
    L = plain_logits(d)
    unfused = mqa.mqa_topk_indices(L, d["ks"], d["ke"], 2048, S_kv=case.S_kv)
    torch.cuda.synchronize()
    assert np.array_equal(got, unfused.cpu().numpy())
    rows = sorted(set(np.linspace(0, case.q.shape[0] - 1, 24).astype(int).tolist()) | {0, 1, 2047})
    rows = [r for r in rows if r < case.q.shape[0]]
    Lr = L[rows].cpu().numpy()
    want = oracle_topk_rows(Lr, case.k_start[rows], case.k_end[rows], 2048, case.S_kv)
    assert np.array_equal(got[rows], want)


def test_captured_in_a_cuda_graph(dev):
    """The call makes no host synchronisation and no allocation, so it can be
    captured in a CUDA graph; replays give the eager result."""
    case = wl.dense_case(96, 12000, 64, 128, seed=995, ranges="causal_tail", clean=False,
                         name="graph")
    d = to_dev(case, dev)
    ws = torch.empty(mqa.mqa_logits_topk_workspace_size(96, 12000), dtype=torch.uint8, device=dev)
    out = torch.full((96, 700), -7, dtype=torch.int32, device=dev)
    eager = fused(d, 700, ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up on the capture stream
        mqa.mqa_logits_topk(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], 700, out,
                            workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mqa.mqa_logits_topk(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], 700, out,
                            workspace=ws)
    for _ in range(3):
        out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), eager)
    assert mqa.device_status() == 0
