"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import build as mqa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mqa.h")


@pytest.fixture(scope="module")
def lib():
    mqa_build.build()
    return mqa.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"MQA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("mqa_logits", "paged_mqa_logits", "paged_mqa_logits_metadata"):
        assert n in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libmqa.so does not export {name}"


def test_library_has_no_cuda_driver_dependency():
    # the driver entry point is fetched at run time: the library loads on a
    # host with no CUDA driver (this container) and links cudart statically
    import subprocess
    out = subprocess.run(["ldd", mqa.library_path()], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart" not in out


def test_status_strings(lib):
    for code, name in mqa.STATUS_NAMES.items():
        assert lib.mqa_status_string(code).decode() == name


F = 16  # a fake, 16-byte aligned "device pointer": never dereferenced on these paths


def call_dense(lib, **kw):
    a = dict(q=F, kv=F, kv_scale=F, weights=F, k_start=F, k_end=F, logits=F, S_q=4, S_kv=256, H=64,
             D=128, ldo=256, flags=1, stream=None)
    a.update(kw)
    return lib.mqa_logits(a["q"], a["kv"], a["kv_scale"], a["weights"], a["k_start"], a["k_end"],
                          a["logits"], a["S_q"], a["S_kv"], a["H"], a["D"], a["ldo"], a["flags"],
                          a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(D=256), 2), (dict(H=16), 2), (dict(H=7), 2),
    (dict(S_q=-1), 1), (dict(S_kv=-5), 1), (dict(ldo=255), 1), (dict(flags=64), 1),
    (dict(flags=3, ldo=0), 1), (dict(q=None), 1), (dict(logits=None), 1),
    (dict(q=F + 8), 1), (dict(kv_scale=F + 4), 1), (dict(logits=F + 2), 1),
    (dict(logits=F + 1, flags=1 | 16), 1), (dict(flags=128), 1), (dict(flags=256), 1),
    (dict(weights=F + 8, flags=1 | 32), 1),
])
def test_dense_rejects_invalid_arguments(lib, kw, status):
    assert call_dense(lib, **kw) == status
    assert lib.mqa_last_error_message().decode()


def test_dense_zero_rows_is_a_no_op(lib):
    assert call_dense(lib, S_q=0, q=None, logits=None) == 0


def call_paged(lib, **kw):
    a = dict(q=F, kv_cache=F, kv_scales=F, weights=F, context_lens=F, block_table=F, max_blocks=16,
             meta=F, logits=F, B=2, next_n=2, H=64, D=128, block_kv=64, num_blocks=40, num_sms=8,
             ldo=1024, flags=1, stream=None)
    a.update(kw)
    return lib.paged_mqa_logits(a["q"], a["kv_cache"], a["kv_scales"], a["weights"],
                                a["context_lens"], a["block_table"], a["max_blocks"], a["meta"],
                                a["logits"], a["B"], a["next_n"], a["H"], a["D"], a["block_kv"],
                                a["num_blocks"], a["num_sms"], a["ldo"], a["flags"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(flags=2), 2), (dict(flags=3), 2), (dict(flags=8), 1), (dict(D=32), 2), (dict(H=8), 2),
    (dict(next_n=65), 2), (dict(block_kv=16), 2), (dict(ldo=1000), 1), (dict(num_sms=0), 1),
    (dict(next_n=0), 1), (dict(B=-1), 1), (dict(meta=None), 1), (dict(kv_cache=F + 1), 1),
    # MQA_KV_FUSED (64): the scales live in the pages, so kv_scales must be NULL
    (dict(flags=1 | 64), 1), (dict(flags=1 | 64 | 2), 2), (dict(flags=1 | 64, kv_scales=None, q=None), 1),
])
def test_paged_rejects_invalid_arguments(lib, kw, status):
    assert call_paged(lib, **kw) == status


def test_paged_zero_batch_is_a_no_op(lib):
    assert call_paged(lib, B=0) == 0


def call_paged_mx(lib, **kw):
    a = dict(q=F, q_sf=F, kv_cache=F, kv_sf=F, weights=F, context_lens=F, block_table=F,
             max_blocks=16, meta=F, logits=F, B=2, next_n=2, H=64, D=128, block_kv=64,
             num_blocks=40, num_sms=8, ldo=1024, flags=1)
    a.update(kw)
    return lib.paged_mqa_logits_mx(a["q"], a["q_sf"], a["kv_cache"], a["kv_sf"], a["weights"],
                                   a["context_lens"], a["block_table"], a["max_blocks"], a["meta"],
                                   a["logits"], a["B"], a["next_n"], a["H"], a["D"], a["block_kv"],
                                   a["num_blocks"], a["num_sms"], a["ldo"], a["flags"], None)


# flags=1 | 8: MXFP4 with the 16-byte aligned fake pointers (32 bytes needed)
@pytest.mark.parametrize("kw,status", [
    (dict(D=64), 2), (dict(q_sf=None), 1), (dict(kv_sf=None), 1), (dict(q_sf=F + 2), 1),
    (dict(flags=1 | 8), 1), (dict(flags=2), 2), (dict(H=8), 2), (dict(block_kv=48), 2),
    (dict(ldo=1000), 1), (dict(flags=1 | 64), 2),
])
def test_paged_mx_rejects_invalid_arguments(lib, kw, status):
    assert call_paged_mx(lib, **kw) == status


@pytest.mark.parametrize("kw,status", [(dict(block_kv=48), 2), (dict(num_sms=0), 1),
                                       (dict(next_n=0), 1), (dict(meta=None), 1)])
def test_metadata_rejects_invalid_arguments(lib, kw, status):
    a = dict(ctx=F, B=3, next_n=2, block_kv=64, num_sms=8, meta=F)
    a.update(kw)
    assert lib.paged_mqa_logits_metadata(a["ctx"], a["B"], a["next_n"], a["block_kv"],
                                         a["num_sms"], a["meta"], None) == status


def test_valid_call_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU suite")
    # passes validation, then the first CUDA runtime call fails: MQA_ERR_CUDA
    assert call_dense(lib) == 3
    assert lib.mqa_get_num_sms(0) == -1


def call_topk(lib, **kw):
    a = dict(logits=F, k_start=F, k_end=F, indices=F, S_q=4, S_kv=256, ldo=256, topk=16, flags=0)
    a.update(kw)
    return lib.mqa_topk_indices(a["logits"], a["k_start"], a["k_end"], a["indices"], a["S_q"],
                                a["S_kv"], a["ldo"], a["topk"], a["flags"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(topk=0), 1), (dict(S_q=-1), 1), (dict(S_kv=-1), 1), (dict(ldo=255), 1),
    (dict(flags=2, ldo=0), 1), (dict(flags=4), 1), (dict(flags=8), 1), (dict(logits=None), 1),
    (dict(indices=None), 1), (dict(k_end=None), 1), (dict(logits=F + 2), 1), (dict(indices=F + 1), 1),
])
def test_topk_rejects_invalid_arguments(lib, kw, status):
    assert call_topk(lib, **kw) == status
    assert lib.mqa_last_error_message().decode()


def test_topk_zero_rows_is_a_no_op(lib):
    assert call_topk(lib, S_q=0, logits=None, indices=None) == 0


def call_paged_topk(lib, **kw):
    a = dict(logits=F, ctx=F, indices=F, B=2, next_n=2, width=1024, ldo=1024, topk=16)
    a.update(kw)
    return lib.paged_mqa_topk_indices(a["logits"], a["ctx"], a["indices"], a["B"], a["next_n"],
                                      a["width"], a["ldo"], a["topk"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(topk=0), 1), (dict(B=-1), 1), (dict(next_n=0), 1), (dict(width=-1), 1),
    (dict(ldo=1000), 1), (dict(ctx=None), 1), (dict(logits=F + 2), 1),
])
def test_paged_topk_rejects_invalid_arguments(lib, kw, status):
    assert call_paged_topk(lib, **kw) == status


def test_paged_topk_zero_batch_is_a_no_op(lib):
    assert call_paged_topk(lib, B=0, logits=None) == 0


def test_valid_topk_call_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU suite")
    assert call_topk(lib) == 3
    assert call_paged_topk(lib) == 3


def test_binding_signatures_match_the_header():
    """Every declared call has a ctypes signature in the binding with the same
    number of parameters (a drift between the two would shift arguments)."""
    import inspect
    text = open(HEADER).read()
    decls = {}
    for m in re.finditer(r"MQA_API\s+[\w\s\*]+?\b(\w+)\s*\(([^)]*)\)", text):
        params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        decls[m.group(1)] = len(params)
    src = inspect.getsource(mqa.load_library)
    sig = dict(re.findall(r'"(\w+)": \(\[([^\]]*)\]', src))
    for name, n in decls.items():
        assert name in sig, f"{name} has no ctypes signature in the binding"
        got = len([a for a in sig[name].split(",") if a.strip()])
        assert got == n, f"{name}: header has {n} parameters, binding {got}"


def call_noalloc(lib, **kw):
    a = dict(q=F, kv_cache=F, kv_scales=F, weights=F, context_lens=F, block_table=F, max_blocks=16,
             logits=F, B=2, next_n=2, H=64, D=128, block_kv=64, num_blocks=40, ldo=1024, flags=1,
             stream=None)
    a.update(kw)
    return lib.paged_mqa_logits_noalloc(a["q"], a["kv_cache"], a["kv_scales"], a["weights"],
                                        a["context_lens"], a["block_table"], a["max_blocks"],
                                        a["logits"], a["B"], a["next_n"], a["H"], a["D"],
                                        a["block_kv"], a["num_blocks"], a["ldo"], a["flags"],
                                        a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(flags=2), 2), (dict(flags=8), 1), (dict(D=32), 2), (dict(H=8), 2),
    (dict(block_kv=16), 2), (dict(ldo=1000), 1), (dict(next_n=0), 1), (dict(B=-1), 1),
    (dict(context_lens=None), 1), (dict(context_lens=F + 2), 1), (dict(logits=None), 1),
    (dict(kv_cache=F + 1), 1), (dict(block_table=F + 2), 1),
])
def test_noalloc_rejects_invalid_arguments_before_any_cuda_call(lib, kw, status):
    # the same host checks as paged_mqa_logits, run before the device is touched
    # (on this GPU-less host a CUDA call would return MQA_ERR_CUDA instead)
    assert call_noalloc(lib, **kw) == status
    assert lib.mqa_last_error_message().decode()


def test_noalloc_zero_batch_is_a_no_op(lib):
    assert call_noalloc(lib, B=0) == 0


def test_metadata_rejects_misaligned_pointers(lib):
    assert lib.paged_mqa_logits_metadata(F + 2, 3, 2, 64, 8, F, None) == 1
    assert lib.paged_mqa_logits_metadata(F, 3, 2, 64, 8, F + 1, None) == 1


@pytest.mark.parametrize("kw,status", [(dict(H=16), 2), (dict(num_sms=0), 1), (dict(S_q=-1), 1),
                                       (dict(meta=None), 1), (dict(ks=F + 2), 1), (dict(meta=F + 1), 1)])
def test_dense_metadata_rejects_invalid_arguments(lib, kw, status):
    a = dict(ks=F, ke=F, S_q=4, S_kv=256, H=64, num_sms=8, meta=F)
    a.update(kw)
    assert lib.mqa_logits_metadata(a["ks"], a["ke"], a["S_q"], a["S_kv"], a["H"], a["num_sms"],
                                   a["meta"], None) == status


def test_scheduled_dense_rejects_invalid_arguments(lib):
    def call(**kw):
        a = dict(meta=F, num_sms=8, D=128)
        a.update(kw)
        return lib.mqa_logits_scheduled(F, F, F, F, F, F, a["meta"], a["num_sms"], F, 4, 256, 64,
                                        a["D"], 256, 1, None)
    assert call(meta=None) == 1
    assert call(D=96) == 2
    assert call(num_sms=0) == 1
    assert call(meta=F + 2) == 1


# flags=1 | 8: MXFP4 with the 16-byte aligned fake pointer, below the 32 bytes
# the packed-E2M1 copies need
@pytest.mark.parametrize("kw,status", [(dict(D=64), 2), (dict(flags=1 | 8), 1), (dict(q_sf=None), 1),
                                       (dict(kv_sf=F + 4), 1), (dict(H=16), 2), (dict(ldo=255), 1)])
def test_mx_rejects_invalid_arguments(lib, kw, status):
    a = dict(q=F, q_sf=F, kv=F, kv_sf=F, D=128, H=64, ldo=256, flags=1)
    a.update(kw)
    assert lib.mqa_logits_mx(a["q"], a["q_sf"], a["kv"], a["kv_sf"], F, F, F, F, 4, 256, a["H"],
                             a["D"], a["ldo"], a["flags"], None) == status


def call_fused(lib, **kw):
    a = dict(q=F, kv=F, kv_scale=F, weights=F, k_start=F, k_end=F, indices=F, ws=256, ws_bytes=1 << 40,
             S_q=4, S_kv=256, H=64, D=128, topk=16, flags=0)
    a.update(kw)
    return lib.mqa_logits_topk(a["q"], a["kv"], a["kv_scale"], a["weights"], a["k_start"], a["k_end"],
                               a["indices"], a["ws"], a["ws_bytes"], a["S_q"], a["S_kv"], a["H"],
                               a["D"], a["topk"], a["flags"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(topk=0), 1), (dict(S_q=-1), 1), (dict(S_kv=-1), 1), (dict(D=96), 2), (dict(H=16), 2),
    (dict(flags=1), 1), (dict(flags=2), 1), (dict(flags=4), 1), (dict(flags=16), 1),
    (dict(q=None), 1), (dict(indices=None), 1), (dict(ws=None), 1), (dict(k_end=None), 1),
    (dict(ws=F), 1), (dict(ws=256 + 64), 1), (dict(indices=F + 2), 1), (dict(q=F + 8), 1),
    (dict(ws_bytes=1000), 1),
])
def test_fused_topk_rejects_invalid_arguments(lib, kw, status):
    assert call_fused(lib, **kw) == status
    assert lib.mqa_last_error_message().decode()


def test_fused_topk_zero_rows_is_a_no_op(lib):
    assert call_fused(lib, S_q=0, q=None, indices=None, ws=None) == 0


def test_fused_topk_workspace_size(lib):
    # one fp32 slot per key (rows padded to 128 keys), one mask word per 32
    # keys (and a scratch row of them), four range words, two thresholds and a
    # selection hint per row, each part 256-aligned
    def r256(x):
        return (x + 255) // 256 * 256
    for S_q, S_kv in ((1, 1), (4, 256), (2048, 32768), (17, 3001), (3, 0)):
        ldo = (max(S_kv, 1) + 127) // 128 * 128
        want = (r256(S_q * ldo * 4) + r256((S_q + 1) * ldo // 32 * 4) + r256(16 * S_q)
                + r256(4 * S_q) + r256(4 * S_q) + r256(4 * S_q))
        assert mqa.mqa_logits_topk_workspace_size(S_q, S_kv) == want
    assert lib.mqa_logits_topk_workspace_size(-1, 5) == 0
