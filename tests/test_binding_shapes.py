"""CPU checks of the binding's shape rules for the paged calls: both
paged_mqa_logits and paged_mqa_logits_noalloc reject inconsistent shapes with
ValueError before anything reaches the library (a wrong row count would
otherwise make the kernel write past the logits)."""
import pytest
import torch

import fp8_mqa_indexer_gb300 as mqa

GOOD = dict(q=(8, 64, 128), kv_cache=(40, 64, 128), kv_scales=(40, 64), weights=(8, 64),
            context_lens=(4,), block_table=(4, 16))


def shapes(**kw):
    a = dict(GOOD)
    a.update(kw)
    return a


def test_consistent_shapes_pass():
    assert mqa.paged_shapes(**GOOD, next_n=2) == (8, 64, 128, 4, 2, 40, 64, 16)
    assert mqa.paged_shapes(**GOOD)[4] == 2          # next_n inferred


def test_fused_page_shapes():
    # kv_scales None: kv_cache [num_blocks, block_kv * (D + 4)] bytes
    fused = dict(GOOD, kv_cache=(40, 64 * 132), kv_scales=None)
    assert mqa.paged_shapes(**fused, next_n=2) == (8, 64, 128, 4, 2, 40, 64, 16)
    with pytest.raises(ValueError):                  # not a whole number of D + 4 rows
        mqa.paged_shapes(**dict(fused, kv_cache=(40, 64 * 132 + 4)), next_n=2)
    with pytest.raises(ValueError):                  # a 3-D cache without scales
        mqa.paged_shapes(**dict(fused, kv_cache=(40, 64, 128)), next_n=2)


@pytest.mark.parametrize("kw", [
    dict(next_n=1),                                  # q rows != B * next_n
    dict(next_n=3),
    dict(block_table=(3, 16)),                       # one table row per sequence
    dict(weights=(8, 32)),
    dict(kv_scales=(40, 32)),
    dict(kv_cache=(40, 64, 64)),                     # D mismatch
    dict(q=(8, 64)),
])
def test_inconsistent_shapes_raise(kw):
    nn = kw.pop("next_n", 2)
    with pytest.raises(ValueError):
        mqa.paged_shapes(**shapes(**kw), next_n=nn)


def _cpu_tensors(**kw):
    s = shapes(**kw)
    u8 = torch.uint8
    return dict(q=torch.zeros(s["q"], dtype=u8), kv_cache=torch.zeros(s["kv_cache"], dtype=u8),
                kv_scales=torch.zeros(s["kv_scales"]), weights=torch.zeros(s["weights"]),
                context_lens=torch.zeros(s["context_lens"], dtype=torch.int32),
                block_table=torch.zeros(s["block_table"], dtype=torch.int32))


@pytest.mark.parametrize("call", ["regular", "noalloc"])
@pytest.mark.parametrize("kw,next_n", [(dict(), 1), (dict(block_table=(5, 16)), 2),
                                        (dict(context_lens=(3,)), 2)])
def test_both_paged_wrappers_reject_bad_shapes(monkeypatch, call, kw, next_n):
    # the device check is bypassed so that the shape rules are what is tested
    monkeypatch.setattr(mqa, "_dev", lambda t, name, dtypes: None)
    monkeypatch.setattr(mqa, "load_library",
                        lambda: pytest.fail("an inconsistent call reached the library"))
    t = _cpu_tensors(**kw)
    out = torch.zeros((8, 1024))
    with pytest.raises(ValueError):
        if call == "regular":
            meta = torch.zeros((9, 2), dtype=torch.int32)
            mqa.paged_mqa_logits(**t, schedule_meta=meta, logits=out, next_n=next_n)
        else:
            mqa.paged_mqa_logits_noalloc(**t, logits=out, next_n=next_n)
