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
