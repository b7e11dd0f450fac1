"""Comparison helpers shared by the GPU parity tests (test infrastructure).

The bar (spec tolerance, restated): masks and ranges bit-exact, every
in-range value within |gpu - ref| <= 1e-3 * sum_h |w * s * x| + 1e-5, where
the right-hand side is computed by the oracle alongside each logit.
"""
from __future__ import annotations

import random
from typing import Iterable, Optional

import numpy as np
import torch


def assert_logits_match(gpu: np.ndarray, ref: np.ndarray, tol: np.ndarray, *, what: str = "",
                        untouched: Optional[np.ndarray] = None) -> None:
    """Compare a slab of GPU logits with the oracle's.

    gpu / ref: float32 [rows, cols]; tol: float64 same shape (0 where ref is not
    a logit).  ``untouched``: boolean mask of positions the call must not have
    written (non-clean mode); there the GPU slab must hold the caller's bytes,
    which ``ref`` carries too.
    """
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    g_inf, r_inf = np.isneginf(gpu), np.isneginf(ref)
    if not np.array_equal(g_inf, r_inf):
        rows, cols = np.nonzero(g_inf != r_inf)
        raise AssertionError(f"{what}: -inf mask differs at {len(rows)} positions, first "
                             f"(row {rows[0]}, col {cols[0]}): gpu={gpu[rows[0], cols[0]]} "
                             f"ref={ref[rows[0], cols[0]]}")
    if untouched is not None:
        same = gpu[untouched].view(np.uint32) == ref[untouched].view(np.uint32)
        assert same.all(), f"{what}: {int((~same).sum())} positions outside the ranges were written"
    logit = np.isfinite(ref)
    if untouched is not None:
        logit &= ~untouched
    g = gpu[logit].astype(np.float64)
    r = ref[logit].astype(np.float64)
    t = tol[logit]
    assert np.isfinite(g).all(), f"{what}: non-finite GPU value where the oracle has a logit"
    err = np.abs(g - r)
    bad = err > t
    if bad.any():
        k = int(np.argmax(err - t))
        rows, cols = np.nonzero(logit)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} logits out of tolerance; "
                             f"worst at (row {rows[k]}, col {cols[k]}): gpu={g[k]!r} ref={r[k]!r} "
                             f"err={err[k]:.3e} tol={t[k]:.3e}")


def sample_rows(n_rows: int, tok: int, extra: int, seed: int = 0) -> list:
    """Rows that cross query-block and 128-row edges, both ends, plus random rows."""
    fixed = {0, 1, tok - 1, tok, 2 * tok - 1, 127, 128, 129, n_rows // 2, n_rows - tok - 1,
             n_rows - tok, n_rows - 2, n_rows - 1}
    rows = {r for r in fixed if 0 <= r < n_rows}
    rng = random.Random(seed)
    while len(rows) < min(n_rows, len(rows) + extra):
        rows.add(rng.randrange(n_rows))
        if len(rows) >= min(n_rows, len(fixed) + extra):
            break
    return sorted(rows)


def dense_valid_mask_gpu(k_start: torch.Tensor, k_end: torch.Tensor, S_kv: int) -> torch.Tensor:
    """Boolean [S_q, S_kv] mask of scored positions, from the ranges alone."""
    cols = torch.arange(S_kv, device=k_start.device, dtype=torch.int64)[None, :]
    lo = k_start.to(torch.int64).clamp(0, S_kv)[:, None]
    hi = k_end.to(torch.int64)[:, None]
    return (cols >= lo) & (cols < hi)


def chunks(n: int, size: int) -> Iterable[tuple]:
    for a in range(0, n, size):
        yield a, min(n, a + size)
