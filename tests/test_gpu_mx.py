"""MXFP8 and MXFP4 dense MQA logits on the GPU (C ABI mqa_logits_mx) against
the CPU oracle's block-scaled definition (oracle_mx_mqa_logits, reading R16).

Masks bit-exact, values within 1e-3 * sum_h |w x| + 1e-5 per logit (x the
block-scaled dot product, computed exactly by the oracle).  The PR #435
reproducer's all-zero input (every scale byte one) must give exact zeros in
range and -inf outside, on the full 2048 x 32768 shape.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import workloads as wl
from parity import assert_logits_match, dense_valid_mask_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU suite needs a CUDA device"
    from fp8_mqa_indexer_gb300 import build
    build.build()
    oracle.build()
    return torch.device("cuda:0")


def upload(case, dev):
    return [t.to(dev) for t in (case.q, case.q_sf, case.kv, case.kv_sf, case.weights, case.k_start,
                                case.k_end)]


def oracle_rows(case, rows, ldo=None, clean=True, compressed=False):
    def one(r):
        return oracle.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                    case.k_start, case.k_end, fp4=case.fp4, ldo=ldo or case.ldo,
                                    clean=clean, compressed=compressed, rows=(r, r + 1),
                                    with_tol=True)
    res = oracle.run_rows_parallel(one, rows)
    return (np.concatenate([res[r][0] for r in rows]), np.concatenate([res[r][1] for r in rows]))


@pytest.mark.parametrize("S_q,S_kv,H,ranges,sf", [
    (129, 1100, 64, "causal_tail", (124, 130)), (64, 700, 64, "full", (110, 140)),
    (150, 900, 32, "causal_tail", (120, 134)), (200, 520, 8, "full", (124, 130)),
    (17, 260, 64, "causal_tail", (127, 127))])
def test_mx_small_full(dev, S_q, S_kv, H, ranges, sf):
    case = wl.mx_dense_case(S_q, S_kv, H, seed=600 + S_q + H, ranges=ranges, sf_lo=sf[0], sf_hi=sf[1])
    out = mqa.mqa_logits_mx(*upload(case, dev))
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    ref, tol = oracle_rows(case, list(range(S_q)))
    assert_logits_match(out.cpu().numpy(), ref, tol, what=f"mx {S_q}x{S_kv} H={H}")


def test_mx_compressed_and_nonclean(dev):
    case = wl.mx_dense_case(70, 600, 64, seed=640, ranges="causal_tail")
    d = upload(case, dev)
    ldo = 600 - 70 + 70
    comp = mqa.mqa_logits_mx(*d, compressed=True, ldo=ldo)
    ref, tol = oracle_rows(case, list(range(70)), ldo=ldo, compressed=True)
    assert_logits_match(comp.cpu().numpy(), ref, tol, what="mx compressed")
    buf = torch.full((70, 600), 5.5, dtype=torch.float32, device=dev)
    mqa.mqa_logits_mx(*d, buf, clean=False)
    got = buf.cpu().numpy()
    ref, tol = oracle_rows(case, list(range(70)))
    inside = np.isfinite(ref)
    assert (got[~inside] == 5.5).all()
    assert np.all(np.abs(got[inside].astype(np.float64) - ref[inside]) <= tol[inside])


def test_mx_unit_scales_match_the_fp8_call(dev):
    """Unit block scales (byte 127) reduce MXFP8 to the FP8 logits with
    kv_scale = 1 (a pin of the oracle, here across the two kernels)."""
    case = wl.mx_dense_case(128, 2048, 64, seed=650, sf_lo=127, sf_hi=127)
    d = upload(case, dev)
    mx = mqa.mqa_logits_mx(*d)
    one = torch.ones(case.S_kv, dtype=torch.float32, device=dev)
    fp8 = mqa.mqa_logits(d[0], d[2], one, d[4], d[5], d[6])
    torch.cuda.synchronize()
    a, b = mx.cpu().numpy(), fp8.cpu().numpy()
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = np.isfinite(b)
    _, tol = oracle_rows(case, list(range(case.S_q)))
    assert np.all(np.abs(a[fin].astype(np.float64) - b[fin]) <= 2 * tol[fin])


@pytest.fixture(scope="module")
def big(dev):
    case = wl.mx_config("mx_2k_32k_h64_d128")
    d = upload(case, dev)
    out = mqa.mqa_logits_mx(*d)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    yield case, d, out
    del d, out
    torch.cuda.empty_cache()


def test_mx_full_size_sampled_rows(big):
    case, d, out = big
    rows = sorted(set(sample_rows(case.S_q, 3, extra=30, seed=7)) | set(range(300, 300 + 64)))
    ref, tol = oracle_rows(case, rows)
    assert_logits_match(out[rows].cpu().numpy(), ref, tol, what=case.name)


def test_mx_full_size_mask_and_determinism(big):
    case, d, out = big
    for a in range(0, case.S_q, 1024):
        valid = dense_valid_mask_gpu(d[5][a:a + 1024], d[6][a:a + 1024], case.S_kv)
        assert torch.equal(out[a:a + 1024].isneginf(), ~valid)
    again = torch.empty_like(out)
    for _ in range(5):
        mqa.mqa_logits_mx(*d, again)
        assert torch.equal(again.view(torch.int32), out.view(torch.int32))


def test_mx_reproducer_all_zero_input(dev):
    """[D] reproducer: all-zero q, k, w with unit scales -> exact zeros in
    [0, KV - Q + row), -inf elsewhere, on the 2048 x 32768 shape."""
    case = wl.mx_config("mx_2k_32k_h64_d128_zeros")
    d = upload(case, dev)
    out = mqa.mqa_logits_mx(*d)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    for a in range(0, case.S_q, 512):
        valid = dense_valid_mask_gpu(d[5][a:a + 512], d[6][a:a + 512], case.S_kv)
        chunk = out[a:a + 512]
        assert torch.equal(chunk.isneginf(), ~valid)
        assert (chunk.masked_fill(~valid, 0) == 0).all()


# ------------------------------------------------------------------ MXFP4
@pytest.mark.parametrize("S_q,S_kv,H,ranges,sf", [
    (129, 1100, 64, "causal_tail", (124, 130)), (64, 700, 64, "full", (110, 140)),
    (150, 900, 32, "causal_tail", (120, 134)), (200, 520, 8, "full", (124, 130)),
    (17, 260, 64, "causal_tail", (127, 127))])
def test_mx4_small_full(dev, S_q, S_kv, H, ranges, sf):
    case = wl.mx_dense_case(S_q, S_kv, H, seed=660 + S_q + H, fp4=True, ranges=ranges,
                            sf_lo=sf[0], sf_hi=sf[1])
    out = mqa.mqa_logits_mx(*upload(case, dev), fp4=True)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    ref, tol = oracle_rows(case, list(range(S_q)))
    assert_logits_match(out.cpu().numpy(), ref, tol, what=f"mxfp4 {S_q}x{S_kv} H={H}")


def test_mx4_compressed_bf16_and_nonclean(dev):
    case = wl.mx_dense_case(70, 600, 64, seed=690, fp4=True, ranges="causal_tail")
    d = upload(case, dev)
    comp = mqa.mqa_logits_mx(*d, compressed=True, ldo=600, fp4=True)
    ref, tol = oracle_rows(case, list(range(70)), ldo=600, compressed=True)
    assert_logits_match(comp.cpu().numpy(), ref, tol, what="mxfp4 compressed")
    f32 = mqa.mqa_logits_mx(*d, fp4=True)
    b16 = mqa.mqa_logits_mx(*d, fp4=True, out_dtype=torch.bfloat16)
    assert torch.equal(b16.view(torch.int16), f32.to(torch.bfloat16).view(torch.int16))
    buf = torch.full((70, 600), 5.5, dtype=torch.float32, device=dev)
    mqa.mqa_logits_mx(*d, buf, clean=False, fp4=True)
    got = buf.cpu().numpy()
    ref, tol = oracle_rows(case, list(range(70)))
    inside = np.isfinite(ref)
    assert (got[~inside] == 5.5).all()
    assert np.all(np.abs(got[inside].astype(np.float64) - ref[inside]) <= tol[inside])


def test_mx4_equals_mx8_of_the_same_values(dev):
    """Every E2M1 value is an E4M3 value: MXFP4 inputs re-encoded as E4M3
    bytes (same scales) give the same logits through the MXFP8 call, up to the
    tensor core's fp32 summation order.  Which nibble is the lower element does
    not matter: q and kv are re-encoded alike."""
    case = wl.mx_dense_case(96, 1500, 64, seed=695, fp4=True, ranges="full")
    tab = torch.tensor(oracle.e2m1_table(), dtype=torch.float32)

    def to_e4m3(packed):
        lo = tab[(packed & 0xF).long()]
        hi = tab[(packed >> 4).long()]
        vals = torch.stack([lo, hi], dim=-1).flatten(-2)
        return vals.to(torch.float8_e4m3fn).view(torch.uint8)

    d4 = upload(case, dev)
    out4 = mqa.mqa_logits_mx(*d4, fp4=True)
    d8 = list(d4)
    d8[0] = to_e4m3(case.q).to(dev)
    d8[2] = to_e4m3(case.kv).to(dev)
    out8 = mqa.mqa_logits_mx(*d8)
    torch.cuda.synchronize()
    _, tol = oracle_rows(case, list(range(case.S_q)))
    a, b = out4.cpu().numpy(), out8.cpu().numpy()
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = np.isfinite(b)
    assert np.all(np.abs(a[fin].astype(np.float64) - b[fin]) <= 2 * tol[fin])


def test_mx4_full_size_sampled_rows_and_determinism(dev):
    case = wl.mx_config("mx4_2k_32k_h64_d128")
    d = upload(case, dev)
    out = mqa.mqa_logits_mx(*d, fp4=True)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    rows = sorted(set(sample_rows(case.S_q, 3, extra=24, seed=9)) | set(range(500, 500 + 32)))
    ref, tol = oracle_rows(case, rows)
    assert_logits_match(out[rows].cpu().numpy(), ref, tol, what=case.name)
    again = torch.empty_like(out)
    for _ in range(3):
        mqa.mqa_logits_mx(*d, again, fp4=True)
        assert torch.equal(again.view(torch.int32), out.view(torch.int32))


def test_mx4_reproducer_all_zero_input(dev):
    """[D] reproducer, MXFP4: all-zero packed q, k and w with unit scales ->
    exact zeros in [0, KV - Q + row), -inf elsewhere, on 2048 x 32768."""
    case = wl.mx_config("mx4_2k_32k_h64_d128_zeros")
    d = upload(case, dev)
    out = mqa.mqa_logits_mx(*d, fp4=True)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    for a in range(0, case.S_q, 512):
        valid = dense_valid_mask_gpu(d[5][a:a + 512], d[6][a:a + 512], case.S_kv)
        chunk = out[a:a + 512]
        assert torch.equal(chunk.isneginf(), ~valid)
        assert (chunk.masked_fill(~valid, 0) == 0).all()
