"""GB300-native MQA logits scoring (the lightning-indexer step).

Thin Python binding over the C ABI of ``libmqa.so`` (declared in
``include/mqa.h``).  Every function here only marshals arguments -- tensor
pointers, sizes, strides, the current CUDA stream -- and calls the library with
the same name; all arithmetic runs in the library's CUDA kernels.  There is no
CPU fallback: if the library is missing or no GPU is present the calls raise.

    logits = mqa_logits(q, kv, kv_scale, weights, k_start, k_end)          # dense
    meta = paged_mqa_logits_metadata(context_lens, next_n=2, block_kv=64)  # paged
    logits = paged_mqa_logits(q, kv_cache, kv_scales, weights, context_lens,
                              block_table, meta)
    idx = mqa_topk_indices(logits, k_start, k_end, topk=2048)      # top-k keys
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

__all__ = [
    "MQAError", "mqa_logits", "mqa_logits_metadata", "mqa_logits_mx", "paged_mqa_logits", "paged_mqa_logits_metadata", "get_num_sms",
    "paged_mqa_logits_noalloc", "paged_mqa_logits_mx", "mqa_topk_indices", "paged_mqa_topk_indices",
    "mqa_logits_topk", "mqa_logits_topk_workspace_size",
    "device_status", "set_wait_limit", "selftest_wait_timeout", "library_path", "load_library",
    "MQA_CLEAN", "MQA_COMPRESSED", "MQA_CHECK_BOUNDS", "MQA_OUT_BF16", "MQA_KV_FUSED",
]

MQA_CLEAN = 1
MQA_COMPRESSED = 2
MQA_CHECK_BOUNDS = 4
MQA_MXFP4 = 8
MQA_OUT_BF16 = 16
MQA_WEIGHTS_BF16 = 32
MQA_KV_FUSED = 64

STATUS_NAMES = {0: "MQA_OK", 1: "MQA_ERR_INVALID_ARG", 2: "MQA_ERR_UNSUPPORTED", 3: "MQA_ERR_CUDA",
                4: "MQA_ERR_TIMEOUT", 5: "MQA_ERR_BAD_INPUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None
_lock = threading.Lock()


class MQAError(RuntimeError):
    """A non-OK ``mqa_status`` from the library."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


def library_path() -> str:
    return os.path.join(_HERE, "libmqa.so")


def load_library() -> ctypes.CDLL:
    """Load libmqa.so (built by ``python -m fp8_mqa_indexer_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m fp8_mqa_indexer_gb300.build`"
                               " (this package has no CPU fallback)")
        lib = ctypes.CDLL(path)
        P, I, I64, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint
        ULL = ctypes.c_ulonglong
        sig = {
            "mqa_logits": ([P, P, P, P, P, P, P, I, I, I, I, I64, U, P], I),
            "mqa_logits_scheduled": ([P, P, P, P, P, P, P, I, P, I, I, I, I, I64, U, P], I),
            "mqa_logits_metadata": ([P, P, I, I, I, I, P, P], I),
            "mqa_logits_mx": ([P, P, P, P, P, P, P, P, I, I, I, I, I64, U, P], I),
            "paged_mqa_logits_metadata": ([P, I, I, I, I, P, P], I),
            "paged_mqa_logits": ([P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, I64, U, P], I),
            "paged_mqa_logits_noalloc": ([P, P, P, P, P, P, I, P, I, I, I, I, I, I, I64, U, P], I),
            "paged_mqa_logits_mx": ([P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, I64, U, P],
                                    I),
            "mqa_topk_indices": ([P, P, P, P, I, I, I64, I, U, P], I),
            "paged_mqa_topk_indices": ([P, P, P, I, I, I, I64, I, P], I),
            "mqa_logits_topk_workspace_size": ([I, I], ctypes.c_size_t),
            "mqa_logits_topk": ([P, P, P, P, P, P, P, P, ctypes.c_size_t, I, I, I, I, I, U, P], I),
            "mqa_get_num_sms": ([I], I),
            "mqa_device_status": ([P], I),
            "mqa_set_wait_limit": ([ULL], I),
            "mqa_selftest_wait_timeout": ([ULL, P], I),
            "mqa_status_string": ([I], ctypes.c_char_p),
            "mqa_last_error_message": ([], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != 0:
        msg = load_library().mqa_last_error_message().decode(errors="replace")
        raise MQAError(status, msg)


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev(t, name: str, dtypes) -> None:
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dense_out(logits, S_q, ldo, compressed, S_kv, out_dtype, device):
    """The [S_q, ldo] output (allocated if None) and its flag bits."""
    import torch
    if logits is None:
        dt = torch.float32 if out_dtype is None else out_dtype
        if dt not in (torch.float32, torch.bfloat16):
            raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
        if ldo is None:
            if compressed:
                raise ValueError("compressed output needs ldo (the longest range) or a logits buffer")
            ldo = S_kv
        logits = torch.empty((S_q, ldo), dtype=dt, device=device)
    else:
        if not (logits.is_cuda and logits.dtype in (torch.float32, torch.bfloat16)
                and logits.dim() == 2 and logits.stride(1) == 1 and logits.shape[0] == S_q):
            raise ValueError("logits must be a CUDA float32 or bfloat16 [S_q, ldo] matrix with unit "
                             "column stride")
        if out_dtype is not None and out_dtype != logits.dtype:
            raise ValueError("out_dtype differs from the logits buffer's dtype")
        ldo = logits.stride(0) if ldo is None else ldo
    return logits, ldo, (MQA_OUT_BF16 if logits.dtype == torch.bfloat16 else 0)


def _fp8_types():
    import torch
    return (torch.float8_e4m3fn, torch.uint8)


def mqa_logits(q, kv, kv_scale, weights, k_start, k_end, logits=None, *, clean: bool = True,
               compressed: bool = False, ldo: Optional[int] = None, check_bounds: bool = False,
               schedule_meta=None, out_dtype=None, stream=None):
    """Dense MQA logits (C ABI ``mqa_logits``, or ``mqa_logits_scheduled`` when
    ``schedule_meta`` from ``mqa_logits_metadata`` is given).

    q [S_q, H, D] and kv [S_kv, D] are E4M3 (float8_e4m3fn or raw uint8 bytes),
    kv_scale [S_kv] float32, weights [S_q, H] float32 or bfloat16 (the flag
    MQA_WEIGHTS_BF16 follows its dtype), k_start / k_end [S_q] int32.
    Returns ``logits`` [S_q, ldo] float32, or bfloat16 with ``out_dtype``
    (allocated when not given; ``ldo`` defaults to S_kv and must be given for
    compressed output).
    """
    import torch
    f8 = _fp8_types()
    _dev(q, "q", f8)
    _dev(kv, "kv", f8)
    _dev(kv_scale, "kv_scale", (torch.float32,))
    _dev(weights, "weights", (torch.float32, torch.bfloat16))
    _dev(k_start, "k_start", (torch.int32,))
    _dev(k_end, "k_end", (torch.int32,))
    S_q, H, D = q.shape
    S_kv = kv.shape[0]
    if kv.dim() != 2 or kv.shape[1] != D or weights.shape != (S_q, H):
        raise ValueError("shape mismatch between q, kv and weights")
    if kv_scale.shape != (S_kv,) or k_start.shape != (S_q,) or k_end.shape != (S_q,):
        raise ValueError("shape mismatch in kv_scale / k_start / k_end")
    logits, ldo, fo = _dense_out(logits, S_q, ldo, compressed, S_kv, out_dtype, q.device)
    flags = (MQA_CLEAN if clean else 0) | (MQA_COMPRESSED if compressed else 0) | \
            (MQA_CHECK_BOUNDS if check_bounds else 0) | fo | _weights_flag(weights)
    with torch.cuda.device(q.device):
        if schedule_meta is None:
            _check(load_library().mqa_logits(_ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(weights),
                                             _ptr(k_start), _ptr(k_end), _ptr(logits), S_q, S_kv,
                                             H, D, ldo, flags, _stream_handle(stream)))
        else:
            _dev(schedule_meta, "schedule_meta", (torch.int32,))
            if schedule_meta.dim() != 2 or schedule_meta.shape[1] != 2:
                raise ValueError("schedule_meta must be an int32 [num_sms + 1, 2] tensor")
            _check(load_library().mqa_logits_scheduled(
                _ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(weights), _ptr(k_start), _ptr(k_end),
                _ptr(schedule_meta), schedule_meta.shape[0] - 1, _ptr(logits), S_q, S_kv, H, D,
                ldo, flags, _stream_handle(stream)))
    return logits


def mqa_logits_mx(q, q_sf, kv, kv_sf, weights, k_start, k_end, logits=None, *, clean: bool = True,
                  compressed: bool = False, ldo: Optional[int] = None, check_bounds: bool = False,
                  out_dtype=None, fp4: bool = False, stream=None):
    """Dense MQA logits with MX inputs (C ABI ``mqa_logits_mx``).

    MXFP8: q [S_q, H, 128] and kv [S_kv, 128] E4M3 (float8_e4m3fn or uint8
    bytes).  ``fp4``: MXFP4, q [S_q, H, 64] and kv [S_kv, 64] bytes (uint8 or
    int8) holding two E2M1 codes each.  q_sf [S_q, H] and kv_sf [S_kv] int32
    (or uint32 bit patterns): four UE8M0 block scales each, byte b for elements
    [32 b, 32 b + 32); weights, ranges and output as ``mqa_logits``.
    """
    import torch
    f8 = (torch.uint8, torch.int8) if fp4 else _fp8_types()
    _dev(q, "q", f8)
    _dev(kv, "kv", f8)
    _dev(q_sf, "q_sf", (torch.int32,))
    _dev(kv_sf, "kv_sf", (torch.int32,))
    _dev(weights, "weights", (torch.float32, torch.bfloat16))
    _dev(k_start, "k_start", (torch.int32,))
    _dev(k_end, "k_end", (torch.int32,))
    if q.dim() != 3 or kv.dim() != 2:
        raise ValueError("q must be [S_q, H, D] and kv [S_kv, D]")
    S_q, H, Db = q.shape
    S_kv = kv.shape[0]
    if kv.shape[1] != Db or weights.shape != (S_q, H) or q_sf.shape != (S_q, H):
        raise ValueError("shape mismatch between q, q_sf, kv and weights")
    if kv_sf.shape != (S_kv,) or k_start.shape != (S_q,) or k_end.shape != (S_q,):
        raise ValueError("shape mismatch in kv_sf / k_start / k_end")
    D = 2 * Db if fp4 else Db   # elements per row
    logits, ldo, fo = _dense_out(logits, S_q, ldo, compressed, S_kv, out_dtype, q.device)
    flags = (MQA_CLEAN if clean else 0) | (MQA_COMPRESSED if compressed else 0) | \
            (MQA_CHECK_BOUNDS if check_bounds else 0) | (MQA_MXFP4 if fp4 else 0) | fo | \
            _weights_flag(weights)
    with torch.cuda.device(q.device):
        _check(load_library().mqa_logits_mx(_ptr(q), _ptr(q_sf), _ptr(kv), _ptr(kv_sf), _ptr(weights),
                                            _ptr(k_start), _ptr(k_end), _ptr(logits), S_q, S_kv, H,
                                            D, ldo, flags, _stream_handle(stream)))
    return logits


def mqa_logits_metadata(k_start, k_end, *, S_kv: int, H: int, num_sms: Optional[int] = None,
                        out=None, stream=None):
    """Dense work schedule (C ABI ``mqa_logits_metadata``): an int32
    [num_sms + 1, 2] tensor of (query block, 128-key tile) start points for
    ``mqa_logits(..., schedule_meta=...)``."""
    import torch
    _dev(k_start, "k_start", (torch.int32,))
    _dev(k_end, "k_end", (torch.int32,))
    if k_start.shape != k_end.shape or k_start.dim() != 1:
        raise ValueError("k_start and k_end must be 1-D of the same length")
    if num_sms is None:
        num_sms = get_num_sms(k_start.device)
    if out is None:
        out = torch.empty((num_sms + 1, 2), dtype=torch.int32, device=k_start.device)
    elif out.shape != (num_sms + 1, 2) or out.dtype != torch.int32 or not out.is_contiguous():
        raise ValueError("schedule_meta must be a contiguous int32 [num_sms + 1, 2] tensor")
    with torch.cuda.device(k_start.device):
        _check(load_library().mqa_logits_metadata(_ptr(k_start), _ptr(k_end), k_start.shape[0],
                                                  S_kv, H, num_sms, _ptr(out),
                                                  _stream_handle(stream)))
    return out


def get_num_sms(device=None) -> int:
    import torch
    dev = torch.cuda.current_device() if device is None else torch.device(device).index or 0
    n = load_library().mqa_get_num_sms(dev)
    if n < 0:
        raise MQAError(3, "cannot query the SM count")
    return n


def paged_mqa_logits_metadata(context_lens, *, next_n: int, block_kv: int,
                              num_sms: Optional[int] = None, out=None, stream=None):
    """Paged work schedule (C ABI ``paged_mqa_logits_metadata``): an int32
    [num_sms + 1, 2] tensor of (sequence, 128-key tile) start points."""
    import torch
    _dev(context_lens, "context_lens", (torch.int32,))
    if num_sms is None:
        num_sms = get_num_sms(context_lens.device)
    if out is None:
        out = torch.empty((num_sms + 1, 2), dtype=torch.int32, device=context_lens.device)
    elif out.shape != (num_sms + 1, 2) or out.dtype != torch.int32 or not out.is_contiguous():
        raise ValueError("schedule_meta must be a contiguous int32 [num_sms + 1, 2] tensor")
    with torch.cuda.device(context_lens.device):
        _check(load_library().paged_mqa_logits_metadata(_ptr(context_lens), context_lens.shape[0],
                                                        next_n, block_kv, num_sms, _ptr(out),
                                                        _stream_handle(stream)))
    return out


def _weights_flag(weights) -> int:
    """MQA_WEIGHTS_BF16 for bf16 weights (fp32 otherwise)."""
    import torch
    return MQA_WEIGHTS_BF16 if weights.dtype == torch.bfloat16 else 0


def _paged_inputs(q, kv_cache, kv_scales, weights, context_lens, block_table, next_n):
    """Type and shape checks shared by the two paged calls; returns
    (R, H, D, B, next_n, num_blocks, block_kv, max_blocks).  kv_scales None:
    the fused layout (kv_cache uint8 [num_blocks, block_kv * (D + 4)])."""
    import torch
    f8 = _fp8_types()
    _dev(q, "q", f8)
    if kv_scales is None:
        _dev(kv_cache, "kv_cache", (torch.uint8,))
    else:
        _dev(kv_cache, "kv_cache", f8)
        _dev(kv_scales, "kv_scales", (torch.float32,))
    _dev(weights, "weights", (torch.float32, torch.bfloat16))
    _dev(context_lens, "context_lens", (torch.int32,))
    _dev(block_table, "block_table", (torch.int32,))
    return paged_shapes(tuple(q.shape), tuple(kv_cache.shape),
                        None if kv_scales is None else tuple(kv_scales.shape),
                        tuple(weights.shape), tuple(context_lens.shape), tuple(block_table.shape),
                        next_n)


def paged_shapes(q, kv_cache, kv_scales, weights, context_lens, block_table, next_n=None):
    """Shape rules of a paged call, on shape tuples alone (no tensors, no GPU).

    Returns (R, H, D, B, next_n, num_blocks, block_kv, max_blocks) or raises
    ValueError: q [B*next_n, H, D], kv_cache [num_blocks, block_kv, D],
    kv_scales [num_blocks, block_kv], weights [B*next_n, H], context_lens [B],
    block_table [B, max_blocks].  kv_scales None: the fused layout, kv_cache
    [num_blocks, block_kv * (D + 4)] bytes.  next_n is inferred from q and
    context_lens when not given.
    """
    fused = kv_scales is None
    if len(q) != 3 or len(kv_cache) != (2 if fused else 3) or len(block_table) != 2 or \
            len(context_lens) != 1:
        raise ValueError("q must be 3-D, kv_cache 3-D (2-D when fused), block_table 2-D, "
                         "context_lens 1-D")
    R, H, D = q
    B = context_lens[0]
    if next_n is None:
        if B == 0 or R % B:
            raise ValueError("cannot infer next_n from q and context_lens")
        next_n = R // B
    if fused:
        num_blocks, page_bytes = kv_cache
        if page_bytes % (D + 4):
            raise ValueError("a fused page holds block_kv * (D + 4) bytes")
        block_kv, D2 = page_bytes // (D + 4), D
    else:
        num_blocks, block_kv, D2 = kv_cache
    if D2 != D or R != B * next_n or tuple(weights) != (R, H) or \
            (not fused and tuple(kv_scales) != (num_blocks, block_kv)):
        raise ValueError("shape mismatch between paged inputs (q rows must be B * next_n)")
    if block_table[0] != B:
        raise ValueError("block_table must have one row per sequence")
    return R, H, D, B, next_n, num_blocks, block_kv, block_table[1]


def _paged_logits_out(logits, R, width, device, out_dtype=None):
    import torch
    if logits is None:
        dt = torch.float32 if out_dtype is None else out_dtype
        if dt not in (torch.float32, torch.bfloat16):
            raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
        return torch.empty((R, width), dtype=dt, device=device)
    if not (isinstance(logits, torch.Tensor) and logits.is_cuda
            and logits.dtype in (torch.float32, torch.bfloat16)
            and logits.dim() == 2 and logits.stride(1) == 1 and logits.shape[0] == R
            and logits.shape[1] >= width):
        raise ValueError("logits must be a CUDA float32 or bfloat16 [B*next_n, >= max_blocks_per_seq"
                         "*block_kv] matrix with unit column stride")
    if out_dtype is not None and out_dtype != logits.dtype:
        raise ValueError("out_dtype differs from the logits buffer's dtype")
    return logits


def paged_mqa_logits(q, kv_cache, kv_scales, weights, context_lens, block_table, schedule_meta,
                     logits=None, *, next_n: Optional[int] = None, clean: bool = True,
                     check_bounds: bool = False, out_dtype=None, stream=None):
    """Paged decode MQA logits (C ABI ``paged_mqa_logits``).

    q [B*next_n, H, D] E4M3, kv_cache [num_blocks, block_kv, D] E4M3, kv_scales
    [num_blocks, block_kv] f32, weights [B*next_n, H] f32, context_lens [B]
    int32, block_table [B, max_blocks_per_seq] int32, schedule_meta from
    ``paged_mqa_logits_metadata``.  Returns logits [B*next_n, ldo] f32 with
    ldo >= max_blocks_per_seq * block_kv.  kv_scales None: the fused page
    layout (flag MQA_KV_FUSED), kv_cache uint8 [num_blocks, block_kv * (D + 4)]
    with each page's key rows followed by their fp32 scales.
    """
    import torch
    R, H, D, B, next_n, num_blocks, block_kv, max_blocks = _paged_inputs(
        q, kv_cache, kv_scales, weights, context_lens, block_table, next_n)
    _dev(schedule_meta, "schedule_meta", (torch.int32,))
    if schedule_meta.dim() != 2 or schedule_meta.shape[1] != 2:
        raise ValueError("schedule_meta must be an int32 [num_sms + 1, 2] tensor")
    num_sms = schedule_meta.shape[0] - 1
    logits = _paged_logits_out(logits, R, max_blocks * block_kv, q.device, out_dtype)
    flags = (MQA_CLEAN if clean else 0) | (MQA_CHECK_BOUNDS if check_bounds else 0) | \
        (MQA_OUT_BF16 if logits.dtype == torch.bfloat16 else 0) | _weights_flag(weights) | \
        (MQA_KV_FUSED if kv_scales is None else 0)
    with torch.cuda.device(q.device):
        _check(load_library().paged_mqa_logits(_ptr(q), _ptr(kv_cache), _ptr(kv_scales), _ptr(weights),
                                               _ptr(context_lens), _ptr(block_table), max_blocks,
                                               _ptr(schedule_meta), _ptr(logits), B, next_n, H, D,
                                               block_kv, num_blocks, num_sms, logits.stride(0), flags,
                                               _stream_handle(stream)))
    return logits


def paged_mqa_logits_mx(q, q_sf, kv_cache, kv_sf, weights, context_lens, block_table,
                        schedule_meta, logits=None, *, next_n: Optional[int] = None,
                        clean: bool = True, check_bounds: bool = False, out_dtype=None,
                        fp4: bool = False, stream=None):
    """Paged decode MQA logits with MX inputs (C ABI ``paged_mqa_logits_mx``).

    MXFP8: q [B*next_n, H, 128] and kv_cache [num_blocks, block_kv, 128] E4M3;
    ``fp4``: MXFP4, q [B*next_n, H, 64] and kv_cache [.., 64] bytes (uint8 or
    int8) of two E2M1 codes.  q_sf [B*next_n, H] and kv_sf [num_blocks,
    block_kv] int32: four UE8M0 scales each.  The rest as ``paged_mqa_logits``.
    """
    import torch
    f8 = (torch.uint8, torch.int8) if fp4 else _fp8_types()
    _dev(q, "q", f8)
    _dev(kv_cache, "kv_cache", f8)
    _dev(q_sf, "q_sf", (torch.int32,))
    _dev(kv_sf, "kv_sf", (torch.int32,))
    _dev(weights, "weights", (torch.float32, torch.bfloat16))
    _dev(context_lens, "context_lens", (torch.int32,))
    _dev(block_table, "block_table", (torch.int32,))
    R, H, Db, B, next_n, num_blocks, block_kv, max_blocks = paged_shapes(
        tuple(q.shape), tuple(kv_cache.shape), tuple(kv_sf.shape), tuple(weights.shape),
        tuple(context_lens.shape), tuple(block_table.shape), next_n)
    if tuple(q_sf.shape) != (R, H):
        raise ValueError("q_sf must be [B*next_n, H]")
    D = 2 * Db if fp4 else Db   # elements per row
    _dev(schedule_meta, "schedule_meta", (torch.int32,))
    if schedule_meta.dim() != 2 or schedule_meta.shape[1] != 2:
        raise ValueError("schedule_meta must be an int32 [num_sms + 1, 2] tensor")
    logits = _paged_logits_out(logits, R, max_blocks * block_kv, q.device, out_dtype)
    flags = (MQA_CLEAN if clean else 0) | (MQA_CHECK_BOUNDS if check_bounds else 0) | \
        (MQA_OUT_BF16 if logits.dtype == torch.bfloat16 else 0) | _weights_flag(weights) | \
        (MQA_MXFP4 if fp4 else 0)
    with torch.cuda.device(q.device):
        _check(load_library().paged_mqa_logits_mx(
            _ptr(q), _ptr(q_sf), _ptr(kv_cache), _ptr(kv_sf), _ptr(weights), _ptr(context_lens),
            _ptr(block_table), max_blocks, _ptr(schedule_meta), _ptr(logits), B, next_n, H, D,
            block_kv, num_blocks, schedule_meta.shape[0] - 1, logits.stride(0), flags,
            _stream_handle(stream)))
    return logits


def paged_mqa_logits_noalloc(q, kv_cache, kv_scales, weights, context_lens, block_table,
                             logits, *, next_n: Optional[int] = None, clean: bool = True,
                             check_bounds: bool = False, stream=None):
    """Paged decode MQA logits with the work schedule kept in the library's own
    fixed device array (C ABI ``paged_mqa_logits_noalloc``): no schedule buffer
    and no allocation.  ``logits`` must be given ([B*next_n, ldo] float32);
    the inputs are checked exactly as for ``paged_mqa_logits`` (kv_scales None:
    the fused page layout)."""
    import torch
    R, H, D, B, next_n, num_blocks, block_kv, max_blocks = _paged_inputs(
        q, kv_cache, kv_scales, weights, context_lens, block_table, next_n)
    if logits is None:
        raise ValueError("paged_mqa_logits_noalloc needs a caller-provided logits buffer")
    logits = _paged_logits_out(logits, R, max_blocks * block_kv, q.device)
    flags = (MQA_CLEAN if clean else 0) | (MQA_CHECK_BOUNDS if check_bounds else 0) | \
        (MQA_OUT_BF16 if logits.dtype == torch.bfloat16 else 0) | _weights_flag(weights) | \
        (MQA_KV_FUSED if kv_scales is None else 0)
    with torch.cuda.device(q.device):
        _check(load_library().paged_mqa_logits_noalloc(
            _ptr(q), _ptr(kv_cache), _ptr(kv_scales), _ptr(weights), _ptr(context_lens),
            _ptr(block_table), max_blocks, _ptr(logits), B, next_n, H, D, block_kv,
            num_blocks, logits.stride(0), flags, _stream_handle(stream)))
    return logits


def _logits_matrix(logits, rows: int) -> None:
    import torch
    if not (isinstance(logits, torch.Tensor) and logits.is_cuda and logits.dtype == torch.float32
            and logits.dim() == 2 and logits.stride(1) == 1 and logits.shape[0] == rows):
        raise ValueError("logits must be a CUDA float32 [rows, ldo] matrix with unit column stride")


def _indices_out(indices, rows: int, topk: int, device):
    import torch
    if indices is None:
        return torch.empty((rows, topk), dtype=torch.int32, device=device)
    if not (indices.is_cuda and indices.dtype == torch.int32 and indices.is_contiguous()
            and tuple(indices.shape) == (rows, topk)):
        raise ValueError("indices must be a contiguous CUDA int32 [rows, topk] tensor")
    return indices


def mqa_topk_indices(logits, k_start, k_end, topk: int, indices=None, *, S_kv: Optional[int] = None,
                     compressed: bool = False, stream=None):
    """Top-k keys per row of dense logits (C ABI ``mqa_topk_indices``).

    ``logits`` [S_q, ldo] float32 (the output of ``mqa_logits``), ``k_start`` /
    ``k_end`` [S_q] int32 (the ranges given to it).  Returns int32 [S_q, topk]:
    the keys with the largest logits in ascending key order, then -1.
    ``S_kv`` (keys of an uncompressed row) defaults to ``ldo``; compressed
    logits need it.
    """
    import torch
    _dev(k_start, "k_start", (torch.int32,))
    _dev(k_end, "k_end", (torch.int32,))
    S_q = k_start.shape[0]
    if k_end.shape != (S_q,):
        raise ValueError("k_start and k_end must have the same length")
    _logits_matrix(logits, S_q)
    ldo = logits.stride(0)
    if S_kv is None:
        if compressed:
            raise ValueError("compressed logits need S_kv (the keys of an uncompressed row)")
        S_kv = logits.shape[1]
    indices = _indices_out(indices, S_q, topk, logits.device)
    flags = MQA_COMPRESSED if compressed else 0
    with torch.cuda.device(logits.device):
        _check(load_library().mqa_topk_indices(_ptr(logits), _ptr(k_start), _ptr(k_end), _ptr(indices),
                                               S_q, S_kv, ldo, topk, flags, _stream_handle(stream)))
    return indices


def mqa_logits_topk_workspace_size(S_q: int, S_kv: int) -> int:
    """Bytes of device workspace ``mqa_logits_topk`` needs for S_q rows of S_kv keys."""
    return int(load_library().mqa_logits_topk_workspace_size(S_q, S_kv))


def mqa_logits_topk(q, kv, kv_scale, weights, k_start, k_end, topk: int, indices=None, *,
                    workspace=None, stream=None):
    """Fused dense logits + top-k (C ABI ``mqa_logits_topk``): the result of
    ``mqa_topk_indices`` over the logits ``mqa_logits`` would compute, without
    writing those logits.  Inputs as ``mqa_logits``; returns int32 [S_q, topk].
    ``workspace``: a CUDA uint8 tensor of at least
    ``mqa_logits_topk_workspace_size(S_q, S_kv)`` bytes (allocated when None).
    """
    import torch
    f8 = _fp8_types()
    _dev(q, "q", f8)
    _dev(kv, "kv", f8)
    _dev(kv_scale, "kv_scale", (torch.float32,))
    _dev(weights, "weights", (torch.float32, torch.bfloat16))
    _dev(k_start, "k_start", (torch.int32,))
    _dev(k_end, "k_end", (torch.int32,))
    S_q, H, D = q.shape
    S_kv = kv.shape[0]
    if kv.dim() != 2 or kv.shape[1] != D or weights.shape != (S_q, H):
        raise ValueError("shape mismatch between q, kv and weights")
    if kv_scale.shape != (S_kv,) or k_start.shape != (S_q,) or k_end.shape != (S_q,):
        raise ValueError("shape mismatch in kv_scale / k_start / k_end")
    need = mqa_logits_topk_workspace_size(S_q, S_kv)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    elif not (isinstance(workspace, torch.Tensor) and workspace.is_cuda
              and workspace.dtype == torch.uint8 and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    indices = _indices_out(indices, S_q, topk, q.device)
    with torch.cuda.device(q.device):
        _check(load_library().mqa_logits_topk(
            _ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(weights), _ptr(k_start), _ptr(k_end),
            _ptr(indices), _ptr(workspace), workspace.numel(), S_q, S_kv, H, D, topk,
            _weights_flag(weights), _stream_handle(stream)))
    return indices


def paged_mqa_topk_indices(logits, context_lens, topk: int, indices=None, *, next_n: int,
                           width: Optional[int] = None, stream=None):
    """Top-k keys per row of paged decode logits (C ABI
    ``paged_mqa_topk_indices``): row b * next_n + t selects among keys
    [0, context_lens[b] - next_n + t + 1).  ``width`` (keys per row) defaults
    to the logits' column count."""
    import torch
    _dev(context_lens, "context_lens", (torch.int32,))
    B = context_lens.shape[0]
    _logits_matrix(logits, B * next_n)
    if width is None:
        width = logits.shape[1]
    indices = _indices_out(indices, B * next_n, topk, logits.device)
    with torch.cuda.device(logits.device):
        _check(load_library().paged_mqa_topk_indices(_ptr(logits), _ptr(context_lens), _ptr(indices),
                                                     B, next_n, width, logits.stride(0), topk,
                                                     _stream_handle(stream)))
    return indices


def device_status(stream=None) -> int:
    """Synchronize and return (and clear) the kernel status word as an
    ``mqa_status`` code (0 = OK, 4 = a wait timed out, 5 = a bounds check failed)."""
    return load_library().mqa_device_status(_stream_handle(stream))


def set_wait_limit(cycles: int) -> None:
    _check(load_library().mqa_set_wait_limit(cycles))


def selftest_wait_timeout(cycles: int, stream=None) -> None:
    _check(load_library().mqa_selftest_wait_timeout(cycles, _stream_handle(stream)))
