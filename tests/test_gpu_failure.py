"""Failure detection on the GPU without a GPU fault: a bounded wait that runs
out returns an error status the host reads, and the context stays usable."""
import pytest
import torch

import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU suite needs a CUDA device"
    from fp8_mqa_indexer_gb300 import build
    build.build()
    return torch.device("cuda:0")


def test_wait_that_nothing_signals_times_out_cleanly(dev):
    assert mqa.device_status() == 0
    mqa.selftest_wait_timeout(2_000_000)        # ~1 ms of SM clock
    assert mqa.device_status() == 4             # MQA_ERR_TIMEOUT, read and cleared
    assert mqa.device_status() == 0
    # the context still runs real work
    case = wl.dense_case(8, 256, 64, 128, seed=500, ranges="full")
    out = mqa.mqa_logits(case.q.to(dev), case.kv.to(dev), case.kv_scale.to(dev),
                         case.weights.to(dev), case.k_start.to(dev), case.k_end.to(dev))
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.isfinite(out).all()


def test_wait_inside_logits_kernel_times_out_drains_and_recovers(dev):
    """A pipeline wait inside the real logits kernel runs out (a budget of a few
    hundred cycles is shorter than any copy from memory): the call reports
    MQA_ERR_TIMEOUT, the kernel's in-flight copies and MMAs are drained before
    it frees its shared memory and TMEM, and the next call, with the default
    budget, matches the oracle."""
    import numpy as np
    import oracle
    from parity import assert_logits_match

    oracle.build()
    case = wl.dense_case(256, 4096, 64, 128, seed=501, ranges="causal_tail")
    args = [t.to(dev) for t in (case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                case.k_end)]
    assert mqa.device_status() == 0
    try:
        mqa.set_wait_limit(300)
        mqa.mqa_logits(*args)
        assert mqa.device_status() == 4         # MQA_ERR_TIMEOUT
    finally:
        mqa.set_wait_limit(0)                   # back to the default budget
    paged = wl.paged_case(3, 2, 64, 128, seed=502, ctx_lo=100, ctx_hi=3000, block_kv=64,
                          num_blocks=200)
    ctx = paged.context_lens.to(dev)
    try:
        mqa.set_wait_limit(300)
        meta = mqa.paged_mqa_logits_metadata(ctx, next_n=2, block_kv=64)
        mqa.paged_mqa_logits(paged.q.to(dev), paged.kv_cache.to(dev), paged.kv_scales.to(dev),
                             paged.weights.to(dev), ctx, paged.block_table.to(dev), meta)
        assert mqa.device_status() == 4
    finally:
        mqa.set_wait_limit(0)
    out = mqa.mqa_logits(*args)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    ref, tol = oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                 case.k_end, with_tol=True)
    assert_logits_match(out.cpu().numpy(), ref, tol, what="after a timed-out call")
    assert np.isneginf(out.cpu().numpy()).any()
