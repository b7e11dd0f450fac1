"""CPU oracle for MQA logits scoring -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``fp8_mqa_indexer_gb300``) never imports, links or calls it, and it never
imports the product library: the two share no code.

The arithmetic lives in ``mqa_oracle.c`` (plain C, double precision, every
function citing the passage of the pages it follows).  This module compiles it
with gcc on first use and exposes it over ctypes with numpy arrays.  ctypes
drops the GIL during a call, so ``*_parallel`` helpers spread independent rows
over host threads without changing any result.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Iterable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mqa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()

CLEAN = 1
COMPRESSED = 2


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, no vendor code)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, u32 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint
            lib.oracle_e4m3_table.argtypes = [P]
            lib.oracle_mqa_logits.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, u32,
                                              i32, i32, P, P]
            lib.oracle_paged_mqa_logits.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                                    i32, i64, u32, i32, i32, P, P]
            lib.oracle_paged_mqa_logits_metadata.argtypes = [P, i32, i32, i32, i32, P]
            lib.oracle_mqa_logits_metadata.argtypes = [P, P, i32, i32, i32, i32, P]
            lib.oracle_topk_indices.argtypes = [P, i64, P, P, i32, i32, u32, i32, i32, i32, P]
            lib.oracle_e2m1_table.argtypes = [P]
            lib.oracle_mx_mqa_logits.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i64,
                                                 u32, i32, i32, P, P]
            lib.oracle_paged_mx_mqa_logits.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                       i32, i32, i32, i32, i64, u32, i32, i32, P, P]
            for f in (lib.oracle_e4m3_table, lib.oracle_mqa_logits, lib.oracle_paged_mqa_logits,
                      lib.oracle_paged_mqa_logits_metadata, lib.oracle_mqa_logits_metadata,
                      lib.oracle_topk_indices,
                      lib.oracle_e2m1_table, lib.oracle_mx_mqa_logits,
                      lib.oracle_paged_mx_mqa_logits):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _np(a, dtype) -> np.ndarray:
    """Contiguous numpy view/copy of a numpy array or CPU torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if str(a.dtype).startswith("torch.float8"):
            import torch
            a = a.view(torch.uint8)
        a = a.numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 E4M3 codes, decoded in double."""
    out = np.empty(256, np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def _flags(clean: bool, compressed: bool) -> int:
    return (CLEAN if clean else 0) | (COMPRESSED if compressed else 0)


def mqa_logits(q, kv, kv_scale, weights, k_start, k_end, *, ldo: Optional[int] = None,
               clean: bool = True, compressed: bool = False,
               rows: Optional[tuple] = None, out: Optional[np.ndarray] = None,
               with_tol: bool = False):
    """Dense MQA logits for rows [r0, r1) (all rows by default).

    q: [S_q, H, D] E4M3 bytes (uint8 or float8 tensor); kv: [S_kv, D] E4M3 bytes;
    kv_scale [S_kv] f32; weights [S_q, H] f32; k_start/k_end [S_q] int32.
    Returns the [r1-r0, ldo] float32 slab (and the float64 tolerance slab if
    ``with_tol``).  ``out`` (pre-filled by the caller) is written in place, which
    is how non-clean mode's untouched positions are observed.
    """
    qn, kvn = _np(q, np.uint8), _np(kv, np.uint8)
    S_q, H, D = qn.shape
    S_kv = kvn.shape[0]
    if ldo is None:
        ldo = S_kv
    r0, r1 = rows if rows is not None else (0, S_q)
    if out is None:
        out = np.full((r1 - r0, ldo), np.nan, np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.shape == (r1 - r0, ldo)
    tol = np.zeros((r1 - r0, ldo), np.float64) if with_tol else None
    sc, w = _np(kv_scale, np.float32), _np(weights, np.float32)
    ks, ke = _np(k_start, np.int32), _np(k_end, np.int32)
    rc = _load().oracle_mqa_logits(_ptr(qn), _ptr(kvn), _ptr(sc), _ptr(w), _ptr(ks), _ptr(ke),
                                   S_q, S_kv, H, D, ldo, _flags(clean, compressed), r0, r1,
                                   _ptr(out), _ptr(tol))
    if rc != 0:
        raise ValueError("oracle_mqa_logits: invalid arguments")
    return (out, tol) if with_tol else out


def paged_mqa_logits(q, kv_cache, kv_scales, weights, context_lens, block_table, *,
                     next_n: int, ldo: Optional[int] = None, clean: bool = True,
                     rows: Optional[tuple] = None, out: Optional[np.ndarray] = None,
                     with_tol: bool = False):
    """Paged decode MQA logits for rows [r0, r1); see ``mqa_oracle.c``."""
    qn = _np(q, np.uint8)
    kvc = _np(kv_cache, np.uint8)
    num_blocks, block_kv, D = kvc.shape
    R, H, D2 = qn.shape
    assert D2 == D
    bt = _np(block_table, np.int32)
    B, max_blocks = bt.shape
    assert R == B * next_n
    width = max_blocks * block_kv
    if ldo is None:
        ldo = width
    r0, r1 = rows if rows is not None else (0, R)
    if out is None:
        out = np.full((r1 - r0, ldo), np.nan, np.float32)
    tol = np.zeros((r1 - r0, ldo), np.float64) if with_tol else None
    sc, w = _np(kv_scales, np.float32), _np(weights, np.float32)
    cl = _np(context_lens, np.int32)
    rc = _load().oracle_paged_mqa_logits(_ptr(qn), _ptr(kvc), _ptr(sc), _ptr(w), _ptr(cl),
                                         _ptr(bt), max_blocks, B, next_n, H, D, block_kv,
                                         num_blocks, ldo, _flags(clean, False), r0, r1,
                                         _ptr(out), _ptr(tol))
    if rc != 0:
        raise ValueError("oracle_paged_mqa_logits: invalid arguments")
    return (out, tol) if with_tol else out


def paged_mqa_logits_metadata(context_lens, *, next_n: int, block_kv: int, num_sms: int) -> np.ndarray:
    """[num_sms + 1, 2] int32 schedule: (sequence, 128-key tile) where each SM starts."""
    cl = _np(context_lens, np.int32)
    meta = np.zeros((num_sms + 1, 2), np.int32)
    rc = _load().oracle_paged_mqa_logits_metadata(_ptr(cl), cl.shape[0], next_n, block_kv,
                                                  num_sms, _ptr(meta))
    if rc != 0:
        raise ValueError("oracle_paged_mqa_logits_metadata: invalid arguments")
    return meta


def mqa_logits_metadata(k_start, k_end, *, S_kv: int, H: int, num_sms: int) -> np.ndarray:
    """[num_sms + 1, 2] int32 dense schedule: (query block, absolute 128-key
    tile) where each SM starts; (num_blocks, 0) at the end."""
    ks = _np(k_start, np.int32)
    ke = _np(k_end, np.int32)
    if ks.shape != ke.shape:
        raise ValueError("k_start and k_end differ in length")
    meta = np.zeros((num_sms + 1, 2), np.int32)
    rc = _load().oracle_mqa_logits_metadata(_ptr(ks), _ptr(ke), ks.shape[0], S_kv, H, num_sms,
                                            _ptr(meta))
    if rc != 0:
        raise ValueError("oracle_mqa_logits_metadata: invalid arguments")
    return meta


def e2m1_table() -> np.ndarray:
    """Value of each of the 16 E2M1 codes, decoded in double."""
    out = np.empty(16, np.float64)
    _load().oracle_e2m1_table(_ptr(out))
    return out


def mx_mqa_logits(q, q_sf, kv, kv_sf, weights, k_start, k_end, *, fp4: bool = False,
                  ldo: Optional[int] = None, clean: bool = True, compressed: bool = False,
                  rows: Optional[tuple] = None, out: Optional[np.ndarray] = None,
                  with_tol: bool = False):
    """MX (block-scaled) dense logits for rows [r0, r1); see ``mqa_oracle.c``.

    q: [S_q, H, 128] E4M3 bytes, or [S_q, H, 64] packed E2M1 bytes when ``fp4``;
    q_sf: [S_q, H] int32/uint32 (four UE8M0 bytes); kv: [S_kv, 128] or [S_kv, 64];
    kv_sf: [S_kv]; weights [S_q, H] f32; k_start/k_end [S_q] int32.
    """
    qn, kvn = _np(q, np.uint8), _np(kv, np.uint8)
    S_q, H, qb = qn.shape
    S_kv = kvn.shape[0]
    D = 2 * qb if fp4 else qb
    if ldo is None:
        ldo = S_kv
    r0, r1 = rows if rows is not None else (0, S_q)
    if out is None:
        out = np.full((r1 - r0, ldo), np.nan, np.float32)
    tol = np.zeros((r1 - r0, ldo), np.float64) if with_tol else None
    qs = np.ascontiguousarray(_np(q_sf, np.int64).astype(np.uint32))
    ks_ = np.ascontiguousarray(_np(kv_sf, np.int64).astype(np.uint32))
    w = _np(weights, np.float32)
    ks, ke = _np(k_start, np.int32), _np(k_end, np.int32)
    rc = _load().oracle_mx_mqa_logits(_ptr(qn), _ptr(qs), _ptr(kvn), _ptr(ks_), _ptr(w), _ptr(ks),
                                      _ptr(ke), S_q, S_kv, H, D, 1 if fp4 else 0, ldo,
                                      _flags(clean, compressed), r0, r1, _ptr(out), _ptr(tol))
    if rc != 0:
        raise ValueError("oracle_mx_mqa_logits: invalid arguments")
    return (out, tol) if with_tol else out


def paged_mx_mqa_logits(q, q_sf, kv_cache, kv_sf, weights, context_lens, block_table, *,
                        next_n: int, fp4: bool = False, ldo: Optional[int] = None,
                        clean: bool = True, rows: Optional[tuple] = None,
                        out: Optional[np.ndarray] = None, with_tol: bool = False):
    """Paged MX logits for rows [r0, r1); see ``mqa_oracle.c``.

    q: [B*next_n, H, 128] E4M3 or [.., 64] packed E2M1 bytes (``fp4``); q_sf
    [B*next_n, H]; kv_cache [num_blocks, block_kv, 128] or [.., 64]; kv_sf
    [num_blocks, block_kv]; weights [B*next_n, H] f32.
    """
    qn, kvc = _np(q, np.uint8), _np(kv_cache, np.uint8)
    R, H, qb = qn.shape
    num_blocks, block_kv, kb = kvc.shape
    assert kb == qb
    D = 2 * qb if fp4 else qb
    bt = _np(block_table, np.int32)
    B, max_blocks = bt.shape
    assert R == B * next_n
    width = max_blocks * block_kv
    if ldo is None:
        ldo = width
    r0, r1 = rows if rows is not None else (0, R)
    if out is None:
        out = np.full((r1 - r0, ldo), np.nan, np.float32)
    tol = np.zeros((r1 - r0, ldo), np.float64) if with_tol else None
    qs = np.ascontiguousarray(_np(q_sf, np.int64).astype(np.uint32))
    ks_ = np.ascontiguousarray(_np(kv_sf, np.int64).astype(np.uint32))
    w = _np(weights, np.float32)
    cl = _np(context_lens, np.int32)
    rc = _load().oracle_paged_mx_mqa_logits(_ptr(qn), _ptr(qs), _ptr(kvc), _ptr(ks_), _ptr(w),
                                            _ptr(cl), _ptr(bt), max_blocks, B, next_n, H, D,
                                            1 if fp4 else 0, block_kv, num_blocks, ldo,
                                            _flags(clean, False), r0, r1, _ptr(out), _ptr(tol))
    if rc != 0:
        raise ValueError("oracle_paged_mx_mqa_logits: invalid arguments")
    return (out, tol) if with_tol else out


def topk_indices(logits, k_start, k_end, *, topk: int, n_cols: Optional[int] = None,
                 compressed: bool = False, rows: Optional[tuple] = None) -> np.ndarray:
    """Top-k keys of rows [r0, r1) of a logits matrix ``[rows, ldo]`` (float32):
    ``[r1 - r0, topk]`` int32, ascending keys then -1; see ``mqa_oracle.c``.

    ``n_cols`` is the number of keys of an uncompressed row (default ``ldo``).
    """
    L = _np(logits, np.float32)
    R, ldo = L.shape
    ks, ke = _np(k_start, np.int32), _np(k_end, np.int32)
    assert ks.shape == (R,) and ke.shape == (R,)
    if n_cols is None:
        n_cols = ldo
    r0, r1 = rows if rows is not None else (0, R)
    out = np.empty((r1 - r0, topk), np.int32)
    rc = _load().oracle_topk_indices(_ptr(L), ldo, _ptr(ks), _ptr(ke), R, n_cols,
                                     COMPRESSED if compressed else 0, topk, r0, r1, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_topk_indices: invalid arguments")
    return out


def paged_ranges(context_lens, next_n: int) -> tuple:
    """Key ranges of the paged decode rows r = b * next_n + t: ``[0, ctx_b -
    next_n + t + 1)`` (empty when negative), as int32 (start, end) arrays."""
    cl = _np(context_lens, np.int64)
    t = np.tile(np.arange(next_n, dtype=np.int64), cl.shape[0])
    end = np.maximum(np.repeat(cl, next_n) - next_n + t + 1, 0)
    return np.zeros(end.shape, np.int32), end.astype(np.int32)


def paged_topk_indices(logits, context_lens, *, next_n: int, topk: int,
                       width: Optional[int] = None, rows: Optional[tuple] = None) -> np.ndarray:
    """Top-k keys of paged decode logits ``[B * next_n, ldo]``; a row has
    ``width`` keys (default ``ldo``)."""
    ks, ke = paged_ranges(context_lens, next_n)
    return topk_indices(logits, ks, ke, topk=topk, n_cols=width, rows=rows)


def _split(rows: Sequence[int], n: int) -> Iterable[list]:
    step = max(1, (len(rows) + n - 1) // n)
    for k in range(0, len(rows), step):
        yield list(rows[k:k + step])


def run_rows_parallel(fn, row_list: Sequence[int], threads: Optional[int] = None) -> dict:
    """Call ``fn(r)`` for every row r over host threads; returns {r: fn(r)}.

    Rows are independent, so the split changes no result.
    """
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    results: dict = {}
    chunks = list(_split(list(row_list), threads))

    def work(chunk):
        for r in chunk:
            results[r] = fn(r)

    ts = [threading.Thread(target=work, args=(c,)) for c in chunks]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return results
