"""bf16 logits (MQA_OUT_BF16) and bf16 weights (MQA_WEIGHTS_BF16) on the GPU,
against the oracle and against the fp32 call.

Reading: a bf16 logit is the fp32 logit rounded to the nearest even bf16,
-inf stays -inf ("[PR #435] ...", section "Validation", lists FP32/BF16
output).  Two checks follow from it: the bf16 output equals the fp32 call's
output rounded by torch's own cast, bit for bit (the kernels share every
step up to the store); and against the oracle, |bf16 - ref| <= tol * (1 + 2^-8)
+ 2^-8 * |ref| (the benchmark spec's tolerance plus half a bf16 ulp, which is at most
2^-8 of the value).
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


def same_as_rounded(bf, f32):
    want = f32.to(torch.bfloat16)
    assert torch.equal(bf.view(torch.int16), want.view(torch.int16))


def check_vs_oracle(bf, ref, tol, what):
    got = bf.float().cpu().numpy()
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), what
    fin = np.isfinite(ref)
    err = np.abs(got[fin].astype(np.float64) - ref[fin])
    bound = tol[fin] * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref[fin])
    assert (err <= bound).all(), f"{what}: {(err > bound).sum()} values out of tolerance"


def dense_args(case, dev):
    return [t.to(dev) for t in (case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                case.k_end)]


@pytest.mark.parametrize("H,D", [(64, 128), (32, 64), (8, 128)])
def test_dense_bf16_small(dev, H, D):
    case = wl.dense_case(129, 1100, H, D, seed=700 + H + D, ranges="causal_tail")
    d = dense_args(case, dev)
    bf = mqa.mqa_logits(*d, out_dtype=torch.bfloat16)
    f32 = mqa.mqa_logits(*d)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert bf.dtype == torch.bfloat16
    same_as_rounded(bf, f32)
    ref, tol = oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                 case.k_end, with_tol=True)
    check_vs_oracle(bf, ref, tol, f"dense bf16 H={H} D={D}")


def test_dense_bf16_compressed_nonclean_and_odd_stride(dev):
    case = wl.dense_case(77, 700, 64, 128, seed=710, ranges="causal_tail")
    d = dense_args(case, dev)
    ldo = 700 - 77 + 77
    bf = mqa.mqa_logits(*d, compressed=True, ldo=ldo, out_dtype=torch.bfloat16)
    f32 = mqa.mqa_logits(*d, compressed=True, ldo=ldo)
    same_as_rounded(bf, f32)
    # non-clean: positions outside the ranges keep the caller's bytes; an odd
    # row stride (in elements) exercises the unaligned fill and store paths
    buf = torch.full((77, 703), 2.5, dtype=torch.bfloat16, device=dev)
    out = mqa.mqa_logits(*d, buf[:, :700], clean=False, ldo=703)
    got = buf.float().cpu().numpy()
    ref, tol = oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                 case.k_end, with_tol=True)
    inside = np.isfinite(ref)
    assert (got[:, :700][~inside] == 2.5).all() and (got[:, 700:] == 2.5).all()
    clean = mqa.mqa_logits(*d, torch.full((77, 703), 2.5, dtype=torch.bfloat16, device=dev)[:, :700],
                           ldo=703)
    check_vs_oracle(clean, ref, tol, "dense bf16 odd stride")
    del out


@pytest.mark.parametrize("next_n,H", [(2, 64), (5, 64), (3, 32)])
def test_paged_bf16_small(dev, next_n, H):
    ctx = [1, 300, 129, 700, 64, 511]
    case = wl.paged_case(6, next_n, H, 128, seed=720 + next_n, ctx_lo=0, ctx_hi=720, block_kv=64,
                         num_blocks=70, context_lens=ctx)
    q, kvc, kvs, w = (case.q.to(dev), case.kv_cache.to(dev), case.kv_scales.to(dev),
                      case.weights.to(dev))
    cl, bt = case.context_lens.to(dev), case.block_table.to(dev)
    meta = mqa.paged_mqa_logits_metadata(cl, next_n=next_n, block_kv=64)
    bf = mqa.paged_mqa_logits(q, kvc, kvs, w, cl, bt, meta, next_n=next_n, out_dtype=torch.bfloat16)
    f32 = mqa.paged_mqa_logits(q, kvc, kvs, w, cl, bt, meta, next_n=next_n)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    same_as_rounded(bf, f32)
    ref, tol = oracle.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, case.weights,
                                       case.context_lens, case.block_table, next_n=next_n,
                                       with_tol=True)
    check_vs_oracle(bf, ref, tol, f"paged bf16 next_n={next_n} H={H}")


def test_mx_bf16_small(dev):
    case = wl.mx_dense_case(100, 900, 64, seed=730)
    d = [t.to(dev) for t in (case.q, case.q_sf, case.kv, case.kv_sf, case.weights, case.k_start,
                             case.k_end)]
    bf = mqa.mqa_logits_mx(*d, out_dtype=torch.bfloat16)
    f32 = mqa.mqa_logits_mx(*d)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    same_as_rounded(bf, f32)


def test_dense_bf16_full_size(dev):
    case = wl.dense_config("dense_2k_32k_h64_d128")
    d = dense_args(case, dev)
    bf = mqa.mqa_logits(*d, out_dtype=torch.bfloat16)
    f32 = mqa.mqa_logits(*d)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    same_as_rounded(bf, f32)


# ------------------------------------------------------------- bf16 weights
# MQA_WEIGHTS_BF16 ("[PR #435] ...", section "Validation": FP32/BF16 weights):
# each weight is widened exactly to fp32, so the call equals the fp32-weight
# call on the same values (the bf16 weights widened by torch) bit for bit,
# and the oracle, given those values, bounds it with the usual tolerance.

def rounded(w):
    return w.to(torch.bfloat16).float()


@pytest.mark.parametrize("H,D", [(64, 128), (32, 64), (8, 128)])
def test_dense_bf16_weights(dev, H, D):
    case = wl.dense_case(131, 1000, H, D, seed=740 + H + D, ranges="causal_tail")
    d = dense_args(case, dev)
    wb = d[3].to(torch.bfloat16)
    got = mqa.mqa_logits(d[0], d[1], d[2], wb, d[4], d[5])
    want = mqa.mqa_logits(d[0], d[1], d[2], wb.float(), d[4], d[5])
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    ref, tol = oracle.mqa_logits(case.q, case.kv, case.kv_scale, rounded(case.weights),
                                 case.k_start, case.k_end, with_tol=True)
    g = got.cpu().numpy()
    assert np.array_equal(np.isneginf(g), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert (np.abs(g[fin].astype(np.float64) - ref[fin]) <= tol[fin]).all()


def test_dense_bf16_weights_scheduled_and_bf16_out(dev):
    case = wl.dense_case(300, 2500, 64, 128, seed=750, ranges="causal_tail")
    d = dense_args(case, dev)
    wb = d[3].to(torch.bfloat16)
    meta = mqa.mqa_logits_metadata(d[4], d[5], S_kv=case.S_kv, H=64)
    a = mqa.mqa_logits(d[0], d[1], d[2], wb, d[4], d[5])
    b = mqa.mqa_logits(d[0], d[1], d[2], wb, d[4], d[5], schedule_meta=meta)
    c = mqa.mqa_logits(d[0], d[1], d[2], wb, d[4], d[5], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    same_as_rounded(c, a)


@pytest.mark.parametrize("fp4", [False, True])
def test_mx_bf16_weights(dev, fp4):
    case = wl.mx_dense_case(100, 700, 64, seed=760 + fp4, fp4=fp4)
    d = [t.to(dev) for t in (case.q, case.q_sf, case.kv, case.kv_sf, case.weights, case.k_start,
                             case.k_end)]
    wb = d[4].to(torch.bfloat16)
    got = mqa.mqa_logits_mx(*d[:4], wb, *d[5:], fp4=fp4)
    want = mqa.mqa_logits_mx(*d[:4], wb.float(), *d[5:], fp4=fp4)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))


@pytest.mark.parametrize("next_n,H", [(2, 64), (5, 64), (4, 16)])
def test_paged_bf16_weights(dev, next_n, H):
    ctx = [1, 300, 129, 700, 64, 511]
    case = wl.paged_case(6, next_n, H, 128, seed=770 + next_n + H, ctx_lo=0, ctx_hi=720,
                         block_kv=64, num_blocks=70, context_lens=ctx)
    q, kvc, kvs, w = (case.q.to(dev), case.kv_cache.to(dev), case.kv_scales.to(dev),
                      case.weights.to(dev))
    cl, bt = case.context_lens.to(dev), case.block_table.to(dev)
    meta = mqa.paged_mqa_logits_metadata(cl, next_n=next_n, block_kv=64)
    wb = w.to(torch.bfloat16)
    got = mqa.paged_mqa_logits(q, kvc, kvs, wb, cl, bt, meta, next_n=next_n)
    want = mqa.paged_mqa_logits(q, kvc, kvs, wb.float(), cl, bt, meta, next_n=next_n)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    ref, tol = oracle.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, rounded(case.weights),
                                       case.context_lens, case.block_table, next_n=next_n,
                                       with_tol=True)
    g = got.cpu().numpy()
    assert np.array_equal(np.isneginf(g), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert (np.abs(g[fin].astype(np.float64) - ref[fin]) <= tol[fin]).all()
