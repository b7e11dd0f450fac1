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


def _timed_out_once(dev, call, attempts=6):
    """Runs `call` with a budget of 100 cycles per wait until one of its waits
    runs out (MQA_ERR_TIMEOUT); the memory it reads is flushed from L2 first,
    so its first copies come from HBM and outlast the budget.  A wait that is
    satisfied within one hardware suspension of mbarrier.try_wait never looks
    at its budget, so a single attempt can complete normally."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(attempts):
        flush.zero_()
        try:
            mqa.set_wait_limit(100)
            call()
            status = mqa.device_status()
        finally:
            mqa.set_wait_limit(0)            # back to the default budget
        assert status in (0, 4)
        if status == 4:
            return True
    return False


def test_wait_inside_logits_kernel_times_out_drains_and_recovers(dev):
    """A pipeline wait inside the real logits kernel runs out: the call reports
    MQA_ERR_TIMEOUT, the kernel's in-flight copies and MMAs are drained before
    it frees its shared memory and TMEM, and the next call, with the default
    budget, matches the oracle."""
    import numpy as np
    import oracle
    from parity import assert_logits_match

    oracle.build()
    case = wl.dense_case(2048, 4096, 64, 128, seed=501, ranges="causal_tail")
    args = [t.to(dev) for t in (case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                case.k_end)]
    assert mqa.device_status() == 0
    assert _timed_out_once(dev, lambda: mqa.mqa_logits(*args))
    paged = wl.paged_case(16, 2, 64, 128, seed=502, ctx_lo=2000, ctx_hi=20000, block_kv=64,
                          num_blocks=6000)
    ctx = paged.context_lens.to(dev)
    pd = [t.to(dev) for t in (paged.q, paged.kv_cache, paged.kv_scales, paged.weights)]
    bt = paged.block_table.to(dev)

    def paged_call():
        meta = mqa.paged_mqa_logits_metadata(ctx, next_n=2, block_kv=64)
        mqa.paged_mqa_logits(*pd, ctx, bt, meta)
    assert _timed_out_once(dev, paged_call)
    # the context still runs real work, with the default budget
    rows = list(range(0, 2048, 7))
    out = mqa.mqa_logits(*args)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    small = wl.dense_case(256, 4096, 64, 128, seed=503, ranges="causal_tail")
    sargs = [t.to(dev) for t in (small.q, small.kv, small.kv_scale, small.weights, small.k_start,
                                 small.k_end)]
    sout = mqa.mqa_logits(*sargs)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    ref, tol = oracle.mqa_logits(small.q, small.kv, small.kv_scale, small.weights, small.k_start,
                                 small.k_end, with_tol=True)
    assert_logits_match(sout.cpu().numpy(), ref, tol, what="after timed-out calls")
    assert torch.isfinite(out[~out.isneginf()]).all()
    del rows
