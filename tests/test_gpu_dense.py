"""Dense MQA logits on the GPU (through the C ABI) against the CPU oracle.

Masks and ranges are compared bit-exactly; values within the oracle's per-logit
tolerance 1e-3 * sum_h |w s x| + 1e-5.  Small workloads are compared in full;
the full-size workloads (2048 x 32768 and 8192 x 65536, H=64, D=128) are
checked on sampled rows against the oracle plus whole-output properties (the
-inf mask from the ranges alone, determinism, row-split and power-of-two
invariance), in the same launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_mqa_indexer_gb300 as mqa
from fp8_mqa_indexer_gb300 import workloads as wl
from parity import assert_logits_match, dense_valid_mask_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the GPU suite needs a CUDA device"
    from fp8_mqa_indexer_gb300 import build
    build.build()
    oracle.build()
    return torch.device("cuda:0")


def upload(case, dev):
    return dict(q=case.q.to(dev), kv=case.kv.to(dev), s=case.kv_scale.to(dev),
                w=case.weights.to(dev), ks=case.k_start.to(dev), ke=case.k_end.to(dev))


def run_gpu(case, d, *, clean=None, compressed=None, out=None, ldo=None, check_bounds=False):
    clean = case.clean if clean is None else clean
    compressed = case.compressed if compressed is None else compressed
    ldo = case.ldo if (ldo is None and out is None) else ldo
    return mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], out, clean=clean,
                          compressed=compressed, ldo=ldo, check_bounds=check_bounds)


def oracle_rows(case, rows, *, clean=None, compressed=None, ldo=None, init=None):
    """Oracle slab for the listed rows (parallel over host threads)."""
    clean = case.clean if clean is None else clean
    compressed = case.compressed if compressed is None else compressed
    ldo = case.ldo if ldo is None else ldo

    def one(r):
        o = None if init is None else init[rows.index(r)][None, :].copy()
        return oracle.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                 case.k_end, ldo=ldo, clean=clean, compressed=compressed,
                                 rows=(r, r + 1), out=o, with_tol=True)

    res = oracle.run_rows_parallel(one, rows)
    ref = np.concatenate([res[r][0] for r in rows])
    tol = np.concatenate([res[r][1] for r in rows])
    return ref, tol


def check_full(case, dev, **kw):
    d = upload(case, dev)
    out = run_gpu(case, d, **kw)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    rows = list(range(case.S_q))
    ref, tol = oracle_rows(case, rows, **{k: v for k, v in kw.items() if k in ("clean", "compressed")})
    assert_logits_match(out.cpu().numpy(), ref, tol, what=case.name)
    return d, out


# ------------------------------------------------------------ full compare
@pytest.mark.parametrize("name", ["dense_tiny", "dense_2k_4k_h32_d64"])
def test_named_small_configs_full(dev, name):
    check_full(wl.dense_config(name), dev)


@pytest.mark.parametrize("H,D", [(8, 64), (8, 128), (32, 64), (32, 128), (64, 64), (64, 128)])
@pytest.mark.parametrize("ranges", ["causal_tail", "suffix"])
def test_head_and_dim_variants(dev, H, D, ranges):
    # non-aligned sizes from the PR #435 validation list (Q=129 / KV=4100) shrunk
    case = wl.dense_case(129, 1100, H, D, seed=200 + H + D, ranges=ranges)
    check_full(case, dev)


def test_nonaligned_pr435_shape(dev):
    check_full(wl.dense_case(129, 4100, 64, 128, seed=301, ranges="causal_tail"), dev)


def test_compact_shape_q17_kv260(dev):
    check_full(wl.dense_case(17, 260, 64, 128, seed=302, ranges="causal_tail"), dev)


def test_irregular_windows_empty_rows_and_clipping(dev):
    g = torch.Generator().manual_seed(7)
    S_q, S_kv = 77, 700
    ks = torch.randint(-50, S_kv + 50, (S_q,), generator=g)
    ln = torch.randint(-20, 400, (S_q,), generator=g)
    ke = ks + ln
    ks[5], ke[5] = 10, 10          # empty
    ks[6], ke[6] = 300, 200        # start > end -> empty
    ks[7], ke[7] = -100, 5000      # clipped to [0, S_kv)
    ks[8], ke[8] = 699, 700        # last key only
    case = wl.dense_case(S_q, S_kv, 64, 128, seed=303, ranges="custom", k_start=ks, k_end=ke)
    check_full(case, dev)


def test_all_zero_inputs_exact(dev):
    """PR #435 reproducer: all-zero Q/K/W -> exactly 0 in range, -inf outside."""
    S_q, S_kv = 129, 4100
    case = wl.dense_case(S_q, S_kv, 64, 128, seed=304, ranges="causal_tail")
    case.q.zero_()
    case.kv.zero_()
    case.weights.zero_()
    d = upload(case, dev)
    out = run_gpu(case, d)
    valid = dense_valid_mask_gpu(d["ks"], d["ke"], S_kv)
    assert torch.equal(out.isneginf(), ~valid)
    assert (out.masked_fill(~valid, 0) == 0).all()


def test_negative_and_zero_scales(dev):
    case = wl.dense_case(64, 520, 64, 128, seed=305, ranges="full")
    g = torch.Generator().manual_seed(3)
    sign = torch.where(torch.rand(case.S_kv, generator=g) < 0.3, -1.0, 1.0)
    case.kv_scale.mul_(sign)
    case.kv_scale[:130] = -case.kv_scale[:130].abs()   # whole warps negative
    case.kv_scale[200:210] = 0.0
    check_full(case, dev)


def test_compressed_small(dev):
    case = wl.dense_case(133, 900, 64, 128, seed=306, ranges="custom",
                         k_start=[(7 * i) % 300 for i in range(133)],
                         k_end=[(7 * i) % 300 + 100 + (i % 450) for i in range(133)],
                         compressed=True)
    check_full(case, dev)


def test_compressed_odd_ldo_and_clipping(dev):
    ks = [-3, 0, 5, 100, 250, 255] * 6
    ke = [40, 255, 6, 90, 257, 255] * 6
    case = wl.dense_case(36, 256, 32, 64, seed=307, ranges="custom", k_start=ks, k_end=ke,
                         compressed=True, ldo=257)
    check_full(case, dev)


def test_nonclean_leaves_outside_untouched(dev):
    case = wl.dense_case(70, 600, 64, 128, seed=308, ranges="suffix")
    d = upload(case, dev)
    sentinel = torch.full((case.S_q, case.S_kv), 12345.5, dtype=torch.float32, device=dev)
    out = run_gpu(case, d, clean=False, out=sentinel)
    assert out.data_ptr() == sentinel.data_ptr()
    rows = list(range(case.S_q))
    init = np.full((case.S_q, case.S_kv), 12345.5, np.float32)
    ref, tol = oracle_rows(case, rows, clean=False, init=[init[r] for r in rows])
    untouched = ~dense_valid_mask_gpu(d["ks"], d["ke"], case.S_kv).cpu().numpy()
    assert_logits_match(out.cpu().numpy(), ref, tol, what="non-clean", untouched=untouched)


def test_row_stride_larger_than_width(dev):
    case = wl.dense_case(40, 300, 32, 128, seed=309, ranges="suffix")
    d = upload(case, dev)
    big = torch.full((case.S_q, 333), 7.0, dtype=torch.float32, device=dev)
    out = run_gpu(case, d, out=big)
    ref, tol = oracle_rows(case, list(range(case.S_q)))
    got = out.cpu().numpy()
    assert_logits_match(got[:, :300].copy(), ref, tol, what="ldo>S_kv")
    assert (got[:, 300:] == 7.0).all(), "columns past S_kv must not be written"


def test_single_key_and_single_row(dev):
    check_full(wl.dense_case(1, 1, 64, 128, seed=310, ranges="full"), dev)
    check_full(wl.dense_case(3, 129, 8, 64, seed=311, ranges="full"), dev)


def test_no_keys(dev):
    case = wl.dense_case(5, 0, 64, 128, seed=312, ranges="full", compressed=True, ldo=7)
    d = upload(case, dev)
    out = run_gpu(case, d)
    assert out.isneginf().all()


# ---------------------------------------------------- full-size workloads
@pytest.fixture(scope="module", params=["dense_2k_32k_h64_d128", "dense_8k_64k_h64_d128",
                                        "dense_8k_64k_h64_d128_compressed"])
def big(dev, request):
    case = wl.dense_config(request.param)
    d = upload(case, dev)
    out = run_gpu(case, d)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    yield case, d, out
    del d, out
    torch.cuda.empty_cache()


def test_full_size_sampled_rows(big):
    case, d, out = big
    rows = sample_rows(case.S_q, 256 // case.H, extra=40, seed=case.S_q)
    # plus every row of one whole query block range of 128 rows
    rows = sorted(set(rows) | set(range(256, 256 + 128)))
    ref, tol = oracle_rows(case, rows)
    got = out[rows].cpu().numpy()
    assert_logits_match(got, ref, tol, what=case.name)


def test_full_size_mask_all_rows(big):
    case, d, out = big
    for a in range(0, case.S_q, 1024):
        b = min(case.S_q, a + 1024)
        sl = out[a:b]
        if case.compressed:
            lens = (d["ke"][a:b].clamp(max=case.S_kv) - d["ks"][a:b].clamp(min=0)).clamp(min=0)
            cols = torch.arange(case.ldo, device=out.device)[None, :]
            valid = cols < lens[:, None]
        else:
            valid = dense_valid_mask_gpu(d["ks"][a:b], d["ke"][a:b], case.S_kv)
        assert torch.equal(sl.isneginf(), ~valid), f"rows {a}..{b}"
        assert torch.isfinite(sl[valid]).all()


def test_full_size_deterministic(big):
    """20 repeats, bitwise ([D] "Validation": 20-repeat bitwise checks)."""
    case, d, out = big
    reps = 20 if case.S_q <= 2048 else 5
    again = torch.empty_like(out)
    for _ in range(reps):
        run_gpu(case, d, out=again, ldo=case.ldo)
        assert torch.equal(again.view(torch.int32), out.view(torch.int32))
    del again


def test_full_size_scheduled_path_is_bitwise_identical(big):
    """The schedule from mqa_logits_metadata (bit-exact against the oracle's)
    gives the same output as the in-kernel split, bit for bit ([D]
    "Validation": scheduled-path equality)."""
    case, d, out = big
    meta = mqa.mqa_logits_metadata(d["ks"], d["ke"], S_kv=case.S_kv, H=case.H)
    want = oracle.mqa_logits_metadata(case.k_start, case.k_end, S_kv=case.S_kv, H=case.H,
                                      num_sms=meta.shape[0] - 1)
    assert np.array_equal(meta.cpu().numpy(), want)
    again = mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], clean=case.clean,
                           compressed=case.compressed, ldo=case.ldo, schedule_meta=meta)
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.equal(again.view(torch.int32), out.view(torch.int32))


def test_full_size_power_of_two_scaling_is_exact(big):
    case, d, out = big
    d2 = dict(d)
    d2["s"] = d["s"] * 2
    d2["w"] = d["w"] * 0.5
    again = run_gpu(case, d2)
    assert torch.equal(again.view(torch.int32), out.view(torch.int32))


def test_full_size_row_split_is_bitwise_identical(big):
    case, d, out = big
    k = 1000  # not a multiple of the query block
    parts = []
    for a, b in ((0, k), (k, case.S_q)):
        sub = {n: d[n][a:b] for n in ("q", "w", "ks", "ke")}
        sub.update(kv=d["kv"], s=d["s"])
        parts.append(mqa.mqa_logits(sub["q"], sub["kv"], sub["s"], sub["w"], sub["ks"], sub["ke"],
                                    clean=case.clean, compressed=case.compressed, ldo=case.ldo))
    whole = torch.cat(parts)
    assert torch.equal(whole.view(torch.int32), out.view(torch.int32))


# ------------------------------------------------------- bounds checking
def test_check_bounds_accepts_valid_input(dev):
    case = wl.dense_case(33, 400, 64, 128, seed=320, ranges="causal_tail")
    d = upload(case, dev)
    out = run_gpu(case, d, check_bounds=True)
    ref, tol = oracle_rows(case, list(range(case.S_q)))
    assert_logits_match(out.cpu().numpy(), ref, tol, what="check-bounds")


@pytest.mark.parametrize("bad", ["start_negative", "end_past_kv", "start_after_end",
                                 "compressed_too_long"])
def test_check_bounds_rejects_bad_ranges(dev, bad):
    case = wl.dense_case(33, 400, 64, 128, seed=321, ranges="causal_tail")
    ks, ke = case.k_start.clone(), case.k_end.clone()
    compressed, ldo = False, None
    if bad == "start_negative":
        ks[3] = -1
    elif bad == "end_past_kv":
        ke[4] = 401
    elif bad == "start_after_end":
        ks[5], ke[5] = 20, 10
    else:
        compressed, ldo = True, 100
    d = upload(case, dev)
    d["ks"], d["ke"] = ks.to(dev), ke.to(dev)
    with pytest.raises(mqa.MQAError) as e:
        mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], compressed=compressed,
                       ldo=ldo or case.ldo, check_bounds=True)
    assert e.value.status == 5
    # and the context is still good
    assert mqa.device_status() == 0
    run_gpu(case, upload(case, dev))
    assert mqa.device_status() == 0


# ------------------------------------------------------- dense schedule
@pytest.mark.parametrize("H,kind,num_sms", [(64, "causal_tail", None), (8, "causal_tail_inclusive", 7),
                                            (32, "suffix", 152), (64, "custom", 5),
                                            (64, "custom", 1000)])
def test_scheduled_equals_unscheduled_and_oracle(dev, H, kind, num_sms):
    ks = ke = None
    if kind == "custom":
        g = torch.Generator().manual_seed(11)
        ks = torch.randint(-30, 900, (150,), generator=g)
        ke = ks + torch.randint(-10, 400, (150,), generator=g)
    case = wl.dense_case(150, 900, H, 128, seed=330 + H, ranges=kind, k_start=ks, k_end=ke)
    d = upload(case, dev)
    meta = mqa.mqa_logits_metadata(d["ks"], d["ke"], S_kv=case.S_kv, H=H, num_sms=num_sms)
    want = oracle.mqa_logits_metadata(case.k_start, case.k_end, S_kv=case.S_kv, H=H,
                                      num_sms=meta.shape[0] - 1)
    assert np.array_equal(meta.cpu().numpy(), want)
    plain = run_gpu(case, d)
    sched = mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], schedule_meta=meta)
    if kind != "custom":   # the custom ranges run past [0, S_kv): the bounds check rejects them
        checked = mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"],
                                 schedule_meta=meta, check_bounds=True)
        assert torch.equal(checked.view(torch.int32), plain.view(torch.int32))
    torch.cuda.synchronize()
    assert mqa.device_status() == 0
    assert torch.equal(sched.view(torch.int32), plain.view(torch.int32))
    ref, tol = oracle_rows(case, list(range(case.S_q)))
    assert_logits_match(sched.cpu().numpy(), ref, tol, what=f"scheduled H={H} {kind}")


def test_scheduled_rejects_a_bad_schedule(dev):
    case = wl.dense_case(150, 900, 64, 128, seed=340, ranges="causal_tail")
    d = upload(case, dev)
    meta = mqa.mqa_logits_metadata(d["ks"], d["ke"], S_kv=case.S_kv, H=64, num_sms=6)
    bad = meta.clone()
    bad[2, 1] += 1
    with pytest.raises(mqa.MQAError) as e:
        mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], schedule_meta=bad,
                       check_bounds=True)
    assert e.value.status == 5
    assert mqa.device_status() == 0
    # without the host check, the kernel's own entry checks refuse a schedule
    # whose slice leaves a block's span, and compute nothing for that slice
    bad2 = meta.clone()
    bad2[1, 1] = 1000
    mqa.mqa_logits(d["q"], d["kv"], d["s"], d["w"], d["ks"], d["ke"], schedule_meta=bad2)
    assert mqa.device_status() == 5
    assert mqa.device_status() == 0
