"""Paged decode MQA logits with MX keys and queries (C ABI paged_mqa_logits_mx)
on the GPU against the CPU oracle's paged MX definition
(oracle_paged_mx_mqa_logits), MXFP8 and MXFP4.

Masks bit-exact, values within 1e-3 * sum_h |w x| + 1e-5 per logit.  Cases:
both element formats, block_kv 32 / 64 / 128, H 16 / 32 / 64, next_n split
into several query atoms (at most 192 / H tokens each), empty and ragged
contexts, bf16 output and weights (bitwise against the fp32 call), unit
scales against the FP8 paged call, and a 64-sequence case with long contexts
on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import workloads as wl
from parity import assert_logits_match

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU suite needs a CUDA device"
    from fp8_mqa_indexer_gb300 import build
    build.build()
    oracle.build()
    return torch.device("cuda:0")


def upload(case, dev):
    return [t.to(dev) for t in (case.q, case.q_sf, case.kv_cache, case.kv_sf, case.weights,
                                case.context_lens, case.block_table)]


def gpu_call(case, d, dev, **kw):
    meta = mqa.paged_mqa_logits_metadata(d[5], next_n=case.next_n, block_kv=case.block_kv)
    out = mqa.paged_mqa_logits_mx(*d, meta, next_n=case.next_n, fp4=case.fp4, **kw)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    return out


def oracle_rows(case, rows):
    def one(r):
        return oracle.paged_mx_mqa_logits(case.q, case.q_sf, case.kv_cache, case.kv_sf,
                                          case.weights, case.context_lens, case.block_table,
                                          next_n=case.next_n, fp4=case.fp4, rows=(r, r + 1),
                                          with_tol=True)
    res = oracle.run_rows_parallel(one, rows)
    return (np.concatenate([res[r][0] for r in rows]), np.concatenate([res[r][1] for r in rows]))


CTX = [1, 0, 300, 129, 700, 64, 511]


@pytest.mark.parametrize("fp4,next_n,H,block_kv", [
    (False, 2, 64, 64), (True, 2, 64, 64), (False, 5, 64, 32), (True, 4, 32, 128),
    (False, 1, 16, 64), (True, 13, 16, 64), (True, 7, 64, 32)])
def test_paged_mx_small(dev, fp4, next_n, H, block_kv):
    case = wl.paged_mx_case(len(CTX), next_n, H, seed=800 + next_n + H + block_kv + fp4,
                            context_lens=CTX, block_kv=block_kv, fp4=fp4)
    out = gpu_call(case, upload(case, dev), dev)
    rows = list(range(case.B * next_n))
    ref, tol = oracle_rows(case, rows)
    assert_logits_match(out.cpu().numpy(), ref, tol,
                        what=f"paged mx fp4={fp4} next_n={next_n} H={H} block_kv={block_kv}")


@pytest.mark.parametrize("fp4", [False, True])
def test_paged_mx_bf16_output_and_weights(dev, fp4):
    case = wl.paged_mx_case(len(CTX), 3, 64, seed=830 + fp4, context_lens=CTX, fp4=fp4)
    d = upload(case, dev)
    f32 = gpu_call(case, d, dev)
    bf = gpu_call(case, d, dev, out_dtype=torch.bfloat16)
    assert torch.equal(bf.view(torch.int16), f32.to(torch.bfloat16).view(torch.int16))
    wb = d[4].to(torch.bfloat16)
    got = gpu_call(case, d[:4] + [wb] + d[5:], dev)
    want = gpu_call(case, d[:4] + [wb.float()] + d[5:], dev)
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))


def test_paged_mx_unit_scales_match_the_fp8_paged_call(dev):
    case = wl.paged_mx_case(len(CTX), 2, 64, seed=840, context_lens=CTX, sf_lo=127, sf_hi=127)
    d = upload(case, dev)
    mx = gpu_call(case, d, dev)
    ones = torch.ones(case.kv_sf.shape, dtype=torch.float32, device=dev)
    meta = mqa.paged_mqa_logits_metadata(d[5], next_n=2, block_kv=case.block_kv)
    fp8 = mqa.paged_mqa_logits(d[0], d[2], ones, d[4], d[5], d[6], meta, next_n=2)
    torch.cuda.synchronize()
    a, b = mx.cpu().numpy(), fp8.cpu().numpy()
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    _, tol = oracle_rows(case, list(range(case.B * 2)))
    fin = np.isfinite(b)
    assert np.all(np.abs(a[fin].astype(np.float64) - b[fin]) <= 2 * tol[fin])


@pytest.mark.parametrize("fp4", [False, True])
def test_paged_mx_long_contexts_sampled(dev, fp4):
    g = torch.Generator().manual_seed(850 + fp4)
    ctx = torch.randint(4096, 32769, (64,), generator=g).tolist()
    case = wl.paged_mx_case(64, 2, 64, seed=851 + fp4, context_lens=ctx, fp4=fp4)
    out = gpu_call(case, upload(case, dev), dev)
    rows = [0, 1, 17, 40, 77, 100, 126, 127]
    ref, tol = oracle_rows(case, rows)
    assert_logits_match(out[rows].cpu().numpy(), ref, tol, what=f"paged mx long fp4={fp4}")
    again = gpu_call(case, upload(case, dev), dev)
    assert torch.equal(again.view(torch.int32), out.view(torch.int32))


@pytest.mark.parametrize("bad", ["block_id", "context", "schedule"])
def test_paged_mx_check_bounds_rejects(dev, bad):
    """MQA_CHECK_BOUNDS: a block id past the pool, a context longer than the
    table's width or a schedule entry out of order is reported as
    MQA_ERR_BAD_INPUT before any logits kernel runs."""
    case = wl.paged_mx_case(4, 2, 64, seed=860, context_lens=[100, 300, 520, 64], fp4=True)
    d = upload(case, dev)
    meta = mqa.paged_mqa_logits_metadata(d[5], next_n=2, block_kv=case.block_kv)
    if bad == "block_id":
        d[6][1, 0] = case.num_blocks
    elif bad == "context":
        d[5][2] = case.max_blocks_per_seq * case.block_kv + 1
    else:
        meta[1, 1] += 1
    with pytest.raises(mqa.MQAError) as e:
        mqa.paged_mqa_logits_mx(*d, meta, next_n=2, fp4=True, check_bounds=True)
    assert e.value.status == 5
    assert mqa.device_status() == 0
    # and a valid call with the check on computes as without it
    good = upload(case, dev)
    meta = mqa.paged_mqa_logits_metadata(good[5], next_n=2, block_kv=case.block_kv)
    a = mqa.paged_mqa_logits_mx(*good, meta, next_n=2, fp4=True, check_bounds=True)
    b = mqa.paged_mqa_logits_mx(*good, meta, next_n=2, fp4=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
