"""Row sharding for running MQA logits on several GPUs (one process per GPU).

Query rows are independent and keys are read-only, so a rank computes a
contiguous slab of rows with the same keys: the inputs it needs are views of
q, weights and the ranges (pointer offsets, no copies), and its output is the
matching slab of the logits.  The top-k selection shards the same way: a
rank selects over its slab of logits rows and ranges and writes the matching
rows of the index matrix.  No collective is needed on the data path; a
caller that wants the whole matrix on one rank gathers the slabs.
"""
from __future__ import annotations


def row_range(n_rows: int, rank: int, world: int, align: int = 1) -> tuple:
    """Balanced contiguous [r0, r1) of rank `rank` out of `world`; inner
    boundaries are multiples of `align` (e.g. a query block)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    units = (n_rows + align - 1) // align
    u0 = units * rank // world
    u1 = units * (rank + 1) // world
    return min(n_rows, u0 * align), min(n_rows, u1 * align)


def dense_row_shard(q, weights, k_start, k_end, rank: int, world: int, align: int = 1):
    """Views of the per-row inputs for this rank's rows, and the row range."""
    r0, r1 = row_range(q.shape[0], rank, world, align)
    return dict(q=q[r0:r1], weights=weights[r0:r1], k_start=k_start[r0:r1],
                k_end=k_end[r0:r1]), (r0, r1)


def topk_row_shard(logits, k_start, k_end, rank: int, world: int):
    """Views of a logits matrix and its ranges for this rank's rows, and the row range."""
    r0, r1 = row_range(logits.shape[0], rank, world)
    return dict(logits=logits[r0:r1], k_start=k_start[r0:r1], k_end=k_end[r0:r1]), (r0, r1)


def paged_sequence_shard(B: int, rank: int, world: int) -> tuple:
    """Contiguous range of sequences [b0, b1) of this rank."""
    return row_range(B, rank, world)
