"""Paged decode MQA logits and the paged work schedule on the GPU (through the
C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import workloads as wl
from parity import assert_logits_match, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU suite needs a CUDA device"
    from fp8_mqa_indexer_gb300 import build
    build.build()
    oracle.build()
    return torch.device("cuda:0")


def upload(case, dev):
    return dict(q=case.q.to(dev), kv=case.kv_cache.to(dev), s=case.kv_scales.to(dev),
                w=case.weights.to(dev), ctx=case.context_lens.to(dev), bt=case.block_table.to(dev))


def run_gpu(case, d, *, num_sms=None, clean=True, out=None, check_bounds=False, meta=None):
    if meta is None:
        meta = mqa.paged_mqa_logits_metadata(d["ctx"], next_n=case.next_n, block_kv=case.block_kv,
                                             num_sms=num_sms)
    return mqa.paged_mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ctx"], d["bt"], meta, out,
                                next_n=case.next_n, clean=clean, check_bounds=check_bounds), meta


def oracle_rows(case, rows, clean=True):
    def one(r):
        return oracle.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, case.weights,
                                       case.context_lens, case.block_table, next_n=case.next_n,
                                       clean=clean, rows=(r, r + 1), with_tol=True)
    res = oracle.run_rows_parallel(one, rows)
    return (np.concatenate([res[r][0] for r in rows]), np.concatenate([res[r][1] for r in rows]))


# ----------------------------------------------------------------- schedule
@pytest.mark.parametrize("B,lo,hi,num_sms", [(64, 4096, 65536, None), (5, 0, 700, 8), (3, 0, 0, 4),
                                             (2000, 0, 3000, 152), (1, 1, 1, 152), (300, 1, 129, 7)])
def test_schedule_matches_oracle_bitwise(dev, B, lo, hi, num_sms):
    g = torch.Generator().manual_seed(B + hi)
    ctx = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)
    n = num_sms or mqa.get_num_sms()
    meta = mqa.paged_mqa_logits_metadata(ctx.to(dev), next_n=2, block_kv=64, num_sms=n)
    want = oracle.paged_mqa_logits_metadata(ctx, next_n=2, block_kv=64, num_sms=n)
    assert np.array_equal(meta.cpu().numpy(), want)


# ------------------------------------------------------------ small, full
@pytest.mark.parametrize("next_n,block_kv,H,D", [
    (2, 64, 64, 128), (1, 64, 64, 128), (4, 64, 64, 128), (3, 32, 32, 128), (2, 128, 64, 128),
    (2, 64, 32, 64), (1, 32, 16, 64), (6, 64, 32, 128), (16, 64, 16, 128),
    # next_n * H above one accumulator (256 columns): query atoms of 256 / H tokens
    (5, 64, 64, 128), (6, 32, 64, 128), (6, 64, 64, 64), (3, 64, 64, 128), (9, 64, 32, 128),
    (20, 128, 16, 128)])
def test_small_paged_full(dev, next_n, block_kv, H, D):
    B = 6
    ctx = [1, next_n - 1, 129, 700, 64, 511]
    case = wl.paged_case(B, next_n, H, D, seed=400 + next_n + block_kv + H, ctx_lo=0, ctx_hi=720,
                         block_kv=block_kv, num_blocks=60, context_lens=ctx)
    d = upload(case, dev)
    for num_sms in (None, 5):
        out, _ = run_gpu(case, d, num_sms=num_sms)
        torch.cuda.synchronize()
        assert mqa.device_status() == 0
        ref, tol = oracle_rows(case, list(range(B * next_n)))
        assert_logits_match(out.cpu().numpy(), ref, tol, what=f"paged n={next_n} bkv={block_kv}")


def test_paged_equals_dense_on_gathered_keys(dev):
    case = wl.paged_case(4, 2, 64, 128, seed=410, ctx_lo=200, ctx_hi=1000, block_kv=64,
                         num_blocks=80)
    d = upload(case, dev)
    paged, _ = run_gpu(case, d)
    for b in range(case.B):
        c = int(case.context_lens[b])
        ids = case.block_table[b, :(c + 63) // 64].long()
        kv = case.kv_cache[ids].reshape(-1, case.D)[:c].contiguous().to(dev)
        s = case.kv_scales[ids].reshape(-1)[:c].contiguous().to(dev)
        rows = slice(2 * b, 2 * b + 2)
        ends = torch.tensor([c - 1, c], dtype=torch.int32, device=dev)
        dense = mqa.mqa_logits(d["q"][rows].contiguous(), kv, s, d["w"][rows].contiguous(),
                               torch.zeros(2, dtype=torch.int32, device=dev), ends)
        ref = dense.cpu().numpy()
        got = paged[rows, :c].cpu().numpy()
        fin = np.isfinite(ref)
        assert np.array_equal(np.isneginf(got), np.isneginf(ref))
        # the same per-key arithmetic: equal up to the MMA's N-dependent order at most
        assert np.allclose(got[fin], ref[fin], rtol=1e-5, atol=1e-5)


def test_paged_nonclean_and_odd_ldo(dev):
    case = wl.paged_case(3, 2, 64, 128, seed=411, ctx_lo=1, ctx_hi=500, block_kv=64, num_blocks=30)
    d = upload(case, dev)
    R, width = 6, case.max_blocks_per_seq * case.block_kv
    buf = torch.full((R, width + 3), 3.25, dtype=torch.float32, device=dev)
    out, _ = run_gpu(case, d, clean=False, out=buf)
    got = out.cpu().numpy()
    assert (got[:, width:] == 3.25).all()
    ref, tol = oracle_rows(case, list(range(R)), clean=True)
    inside = np.isfinite(ref)
    assert (got[:, :width][~inside] == 3.25).all()
    g = got[:, :width]
    assert np.all(np.abs(g[inside] - ref[inside]) <= tol[inside])


# ---------------------------------------------------------- full size
@pytest.fixture(scope="module")
def big(dev):
    case = wl.paged_config("paged_b64_n2_h64_d128")
    d = upload(case, dev)
    out, meta = run_gpu(case, d)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    yield case, d, out, meta
    del d, out
    torch.cuda.empty_cache()


def test_full_size_paged_sampled_rows(big):
    case, d, out, meta = big
    rows = sample_rows(case.B * case.next_n, case.next_n, extra=24, seed=5)
    ref, tol = oracle_rows(case, rows)
    assert_logits_match(out[rows].cpu().numpy(), ref, tol, what=case.name)


def test_full_size_paged_mask(big):
    case, d, out, meta = big
    width = case.max_blocks_per_seq * case.block_kv
    ends = d["ctx"].to(torch.int64).repeat_interleave(case.next_n) - case.next_n + \
        torch.arange(case.next_n, device=out.device).repeat(case.B) + 1
    cols = torch.arange(width, device=out.device)[None, :]
    valid = cols < ends[:, None]
    assert torch.equal(out.isneginf(), ~valid)
    assert torch.isfinite(out[valid]).all()


def test_full_size_paged_deterministic(big):
    case, d, out, meta = big
    again, _ = run_gpu(case, d, meta=meta)
    assert torch.equal(again.view(torch.int32), out.view(torch.int32))


def test_full_size_paged_schedule(big):
    case, d, out, meta = big
    want = oracle.paged_mqa_logits_metadata(case.context_lens, next_n=case.next_n,
                                            block_kv=case.block_kv, num_sms=meta.shape[0] - 1)
    assert np.array_equal(meta.cpu().numpy(), want)


# ------------------------------------------------------- bounds checking
@pytest.mark.parametrize("bad", ["block_id", "context", "schedule"])
def test_paged_check_bounds_rejects(dev, bad):
    case = wl.paged_case(4, 2, 64, 128, seed=420, ctx_lo=100, ctx_hi=600, block_kv=64, num_blocks=40)
    d = upload(case, dev)
    meta = mqa.paged_mqa_logits_metadata(d["ctx"], next_n=2, block_kv=64)
    if bad == "block_id":
        d["bt"][1, 0] = 40
    elif bad == "context":
        d["ctx"][2] = case.max_blocks_per_seq * 64 + 1
    else:
        meta[1, 1] += 1
    with pytest.raises(mqa.MQAError) as e:
        run_gpu(case, d, check_bounds=True, meta=meta)
    assert e.value.status == 5
    assert mqa.device_status() == 0


def test_paged_check_bounds_accepts_valid(dev):
    case = wl.paged_case(4, 2, 64, 128, seed=421, ctx_lo=100, ctx_hi=600, block_kv=64, num_blocks=40)
    d = upload(case, dev)
    out, _ = run_gpu(case, d, check_bounds=True)
    ref, tol = oracle_rows(case, list(range(8)))
    assert_logits_match(out.cpu().numpy(), ref, tol, what="paged check-bounds")
