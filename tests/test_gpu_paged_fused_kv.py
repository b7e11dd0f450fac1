"""Paged decode logits with the fused page layout (MQA_KV_FUSED: each page
holds its block_kv key rows, then their block_kv fp32 scales) on the GPU,
through the C ABI.

The fused layout carries the same keys and scales as the separate
`kv_cache` / `kv_scales` tensors, so every case checks the fused call bit for
bit against the separate-layout call on the same data, and against the CPU
oracle (run on the separate tensors) within the logits tolerance.  Cases cover
block_kv 32 / 64 / 128, D 64 / 128, H 16 / 32 / 64, next_n up to 6, contexts
of 0, 1 and ragged lengths, non-clean output, bf16 logits and weights, the
no-allocation call, bounds checking and the 64-sequence decode workload.
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


def fuse(kv_cache, kv_scales):
    """[num_blocks, block_kv * (D + 4)] bytes: each page's key rows, then its scales."""
    nb, bkv, D = kv_cache.shape
    keys = kv_cache.contiguous().view(torch.uint8).reshape(nb, bkv * D)
    scales = kv_scales.contiguous().view(torch.uint8).reshape(nb, bkv * 4)
    return torch.cat([keys, scales], dim=1).contiguous()


def upload(case, dev):
    return dict(q=case.q.to(dev), kv=case.kv_cache.to(dev), s=case.kv_scales.to(dev),
                fused=fuse(case.kv_cache, case.kv_scales).to(dev), w=case.weights.to(dev),
                ctx=case.context_lens.to(dev), bt=case.block_table.to(dev))


def both(case, d, **kw):
    meta = mqa.paged_mqa_logits_metadata(d["ctx"], next_n=case.next_n, block_kv=case.block_kv)
    sep = mqa.paged_mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ctx"], d["bt"], meta,
                               next_n=case.next_n, **kw)
    fus = mqa.paged_mqa_logits(d["q"], d["fused"], None, d["w"], d["ctx"], d["bt"], meta,
                               next_n=case.next_n, **kw)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    return sep, fus


def check_oracle(case, out, clean=True):
    R = case.q.shape[0]
    ref, tol = oracle.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, case.weights,
                                       case.context_lens, case.block_table, next_n=case.next_n,
                                       clean=clean, with_tol=True)
    got = out.float().cpu().numpy()[:, :ref.shape[1]]
    assert_logits_match(got[:R], ref, tol, what="fused pages")


@pytest.mark.parametrize("next_n,block_kv,H,D", [
    (2, 64, 64, 128), (1, 32, 64, 128), (2, 128, 64, 128), (3, 32, 32, 128), (2, 64, 32, 64),
    (1, 32, 16, 64), (6, 64, 64, 128), (5, 128, 16, 64)])
def test_fused_pages_equal_separate_pages(dev, next_n, block_kv, H, D):
    ctx = [1, 0, 129, 700, 64, 511, next_n]
    case = wl.paged_case(len(ctx), next_n, H, D, seed=1400 + next_n + block_kv + H + D, ctx_lo=0,
                         ctx_hi=720, block_kv=block_kv, num_blocks=80, context_lens=ctx)
    d = upload(case, dev)
    sep, fus = both(case, d)
    assert torch.equal(sep.view(torch.int32), fus.view(torch.int32))
    check_oracle(case, fus)


def test_fused_pages_nonclean_bf16(dev):
    case = wl.paged_case(5, 2, 64, 128, seed=1450, ctx_lo=10, ctx_hi=900, block_kv=64,
                         num_blocks=90)
    d = upload(case, dev)
    sep, fus = both(case, d, clean=False)
    # untouched positions hold whatever the fresh buffers held: compare the scored ones
    R, width = sep.shape
    ks, ke = oracle.paged_ranges(case.context_lens, 2)
    for r in range(R):
        assert torch.equal(sep[r, :ke[r]].view(torch.int32), fus[r, :ke[r]].view(torch.int32))
    d["w"] = d["w"].bfloat16()
    sep, fus = both(case, d, out_dtype=torch.bfloat16)
    assert torch.equal(sep.view(torch.int16), fus.view(torch.int16))


def test_fused_pages_noalloc_and_bounds(dev):
    case = wl.paged_case(4, 2, 64, 128, seed=1460, ctx_lo=100, ctx_hi=600, block_kv=64,
                         num_blocks=40)
    d = upload(case, dev)
    sep, fus = both(case, d)
    out = torch.empty_like(fus)
    mqa.paged_mqa_logits_noalloc(d["q"], d["fused"], None, d["w"], d["ctx"], d["bt"], out,
                                 next_n=2)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.equal(out.view(torch.int32), fus.view(torch.int32))
    # a block id past the pool is rejected under bounds checking
    bad = d["bt"].clone()
    bad[1, 0] = 40
    meta = mqa.paged_mqa_logits_metadata(d["ctx"], next_n=2, block_kv=64)
    with pytest.raises(mqa.MQAError):
        mqa.paged_mqa_logits(d["q"], d["fused"], None, d["w"], d["ctx"], bad, meta, next_n=2,
                             check_bounds=True)
    assert mqa.device_status() == 0


def test_fused_pages_decode_workload(dev):
    """The 64-sequence decode workload: fused equals separate on every row."""
    case = wl.paged_config("paged_b64_n2_h64_d128")
    d = upload(case, dev)
    sep, fus = both(case, d)
    assert torch.equal(sep.view(torch.int32), fus.view(torch.int32))
