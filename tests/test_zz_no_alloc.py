"""The no-allocation paged decode call, against the regular one.

paged_mqa_logits_noalloc is for callers that cannot allocate device memory (a
C program or plugin without access to the allocator that owns the GPU, a
decode loop that must not risk the device synchronization cudaMalloc may
cause, a service with a fixed memory plan).  It keeps the work schedule in a
fixed array inside the library instead of a caller buffer.  Two calls in a
row, with different context lengths, must each match the regular
paged_mqa_logits call (schedule from paged_mqa_logits_metadata in a caller
buffer) within the parity tolerance of the other GPU tests, with identical
-inf masks.  This file sorts last so that a failure here stops a run only
after every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _case(seed, ctx):
    return wl.paged_case(len(ctx), 2, 64, 128, seed=seed, ctx_lo=1, ctx_hi=1500, block_kv=64,
                         num_blocks=200, context_lens=ctx)


def test_noalloc_matches_regular_call_twice_in_a_row():
    assert torch.cuda.is_available(), "the GPU suite needs a CUDA device"
    from fp8_mqa_indexer_gb300 import build
    build.build()
    oracle.build()
    dev = torch.device("cuda:0")
    for seed, ctx in ((801, [1500, 3, 700, 129, 64, 1000]), (802, [5, 1200, 1499, 2])):
        case = _case(seed, ctx)
        q, kvc, kvs = case.q.to(dev), case.kv_cache.to(dev), case.kv_scales.to(dev)
        w, cl, bt = case.weights.to(dev), case.context_lens.to(dev), case.block_table.to(dev)
        R = case.B * case.next_n
        width = case.max_blocks_per_seq * case.block_kv
        meta = mqa.paged_mqa_logits_metadata(cl, next_n=2, block_kv=64)
        ref = mqa.paged_mqa_logits(q, kvc, kvs, w, cl, bt, meta, next_n=2)
        out = torch.full((R, width), 7.0, dtype=torch.float32, device=dev)
        mqa.paged_mqa_logits_noalloc(q, kvc, kvs, w, cl, bt, out, next_n=2)
        torch.cuda.synchronize()
        assert mqa.device_status() == 0
        _, tol = oracle.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, case.weights,
                                         case.context_lens, case.block_table, next_n=2,
                                         with_tol=True)
        a, b = out.cpu().numpy(), ref.cpu().numpy()
        assert np.array_equal(np.isneginf(a), np.isneginf(b))
        fin = np.isfinite(b)
        assert np.isfinite(a[fin]).all()
        assert (np.abs(a[fin].astype(np.float64) - b[fin]) <= tol[fin]).all()

    # The property the call exists for: once warmed up (kernels loaded, the
    # array's address looked up), a call allocates no device memory, neither
    # through torch's allocator nor through the driver.
    torch.cuda.synchronize()
    allocs0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    free0 = torch.cuda.mem_get_info()[0]
    mqa.paged_mqa_logits_noalloc(q, kvc, kvs, w, cl, bt, out, next_n=2)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs0
    assert torch.cuda.mem_get_info()[0] == free0
