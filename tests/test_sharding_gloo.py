"""Multi-rank path on CPU: two gloo ranks each score their row slab (views of
the inputs, same keys) with the oracle, and each selects the top-k keys of its
slab of logits rows; the gathered slabs must equal the unsharded results bit
for bit, and the split must cover every row once."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp8_mqa_indexer_gb300 import sharding


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    import oracle
    from fp8_mqa_indexer_gb300 import workloads as wl
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = wl.dense_case(37, 300, 8, 64, seed=901, ranges="causal_tail_inclusive")
    views, (r0, r1) = sharding.dense_row_shard(case.q, case.weights, case.k_start, case.k_end,
                                              rank, world)
    slab = oracle.mqa_logits(views["q"], case.kv, case.kv_scale, views["weights"],
                             views["k_start"], views["k_end"], ldo=case.S_kv)
    slabs = [None] * world
    dist.all_gather_object(slabs, (r0, r1, slab))
    # the benchmark's aggregation: the slowest rank's time
    t = torch.tensor([float(rank + 1)])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        full = oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                 case.k_end)
        rows = sorted(slabs, key=lambda s: s[0])
        got = np.concatenate([s[2] for s in rows])
        ok = (np.array_equal(got.view(np.uint32), full.view(np.uint32))
              and [s[0] for s in rows] == [0, rows[0][1]] and rows[-1][1] == case.S_q
              and float(t.item()) == float(world))
        with open(result_path, "w") as f:
            f.write("ok" if ok else "mismatch")
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_row_sharding_is_bitwise(tmp_path):
    import oracle
    oracle.build()
    out = tmp_path / "result.txt"
    mp.start_processes(_worker, args=(2, _free_port(), str(out)), nprocs=2, start_method="spawn")
    assert out.read_text() == "ok"


def _topk_worker(rank, world, port, result_path):
    import oracle
    from fp8_mqa_indexer_gb300 import workloads as wl
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = wl.topk_case(41, 900, 50, seed=902, ranges="causal_tail", levels=3)
    views, (r0, r1) = sharding.topk_row_shard(case.logits, case.k_start, case.k_end, rank, world)
    slab = oracle.topk_indices(views["logits"], views["k_start"], views["k_end"], topk=case.topk,
                               n_cols=case.n_cols)
    slabs = [None] * world
    dist.all_gather_object(slabs, (r0, r1, slab))
    if rank == 0:
        full = oracle.topk_indices(case.logits, case.k_start, case.k_end, topk=case.topk,
                                   n_cols=case.n_cols)
        rows = sorted(slabs, key=lambda s: s[0])
        got = np.concatenate([s[2] for s in rows])
        ok = np.array_equal(got, full) and rows[0][0] == 0 and rows[-1][1] == case.rows
        with open(result_path, "w") as f:
            f.write("ok" if ok else "mismatch")
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_topk_sharding_is_bitwise(tmp_path):
    import oracle
    oracle.build()
    out = tmp_path / "result.txt"
    mp.start_processes(_topk_worker, args=(2, _free_port(), str(out)), nprocs=2, start_method="spawn")
    assert out.read_text() == "ok"


@pytest.mark.parametrize("n,world,align", [(37, 2, 1), (2048, 3, 4), (5, 8, 1), (0, 2, 1),
                                           (8192, 8, 4)])
def test_row_ranges_partition_rows(n, world, align):
    ranges = [sharding.row_range(n, r, world, align) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0 and a0 <= a1
    for a0, _ in ranges[1:]:
        assert a0 % align == 0 or a0 == n
