"""Pins for the oracle's MX (block-scaled) logits, independent of its code.

The MX variant is the one the "[PR #435] Improve SM100 MX MQA logits
clean-output performance" page times: E4M3 (MXFP8) or packed E2M1 (MXFP4)
elements, four UE8M0 block scales per 128-element row packed in an int32,
0x7f7f7f7f meaning every scale is one.  Pinned here by: the E2M1 format's
eight magnitudes written as literals; the reproducer's all-zero check (exact
zeros in range, -inf outside); unit scales reducing MXFP8 to the pinned FP8
logits with kv_scale = 1; one head with unit weights reducing to torch.matmul
in float64 on decoded, scaled values; exact power-of-two scaling per block;
hand-derived block-to-byte cases; the nibble order being unobservable.  The
paged MX oracle is pinned bit for bit to the dense one over keys gathered
through the block table by tensor indexing, to the paged FP8 oracle by unit
scales, and by a hand case.
"""
import numpy as np
import pytest
import torch

from fp8_mqa_indexer_gb300 import workloads as wl

ONE = 0x7F7F7F7F   # four UE8M0 bytes of 127: every block scale is 2^0


def e2m1_literal():
    """E2M1 magnitudes for codes 0..7 (exponent bits, mantissa bit), then negatives."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    return np.array(mags + [-m for m in mags])


def sf(*bytes4):
    v = bytes4[0] | (bytes4[1] << 8) | (bytes4[2] << 16) | (bytes4[3] << 24)
    return v - (1 << 32) if v >= 1 << 31 else v


def decode_scaled(case, which):
    """float64 [rows, 128] of decoded elements times their block scales (torch/numpy only)."""
    data = case.q if which == "q" else case.kv
    scales = case.q_sf if which == "q" else case.kv_sf
    if case.fp4:
        tab = torch.tensor(e2m1_literal())
        lo, hi = (data & 0xF).long(), (data >> 4).long()
        vals = torch.stack([tab[lo], tab[hi]], dim=-1).reshape(*data.shape[:-1], 128)
    else:
        vals = data.view(torch.float8_e4m3fn).to(torch.float64)
    s = scales.to(torch.int64) & 0xFFFFFFFF
    exps = torch.stack([(s >> (8 * b)) & 0xFF for b in range(4)], dim=-1).to(torch.float64)
    mult = torch.repeat_interleave(torch.pow(2.0, exps - 127), 32, dim=-1)
    return vals * mult


def test_e2m1_table_matches_format_literals(oracle_mod):
    tab = oracle_mod.e2m1_table()
    want = e2m1_literal()
    assert np.array_equal(tab, want) and np.array_equal(np.signbit(tab), np.signbit(want))


@pytest.mark.parametrize("fp4", [False, True])
def test_all_zero_inputs_give_zero_and_neg_inf(oracle_mod, fp4):
    # the PR #435 reproducer: all-zero q, k and weights, unit scales, rows [0, KV - Q + row)
    S_q, S_kv, H = 16, 96, 4
    nb = 64 if fp4 else 128
    q = torch.zeros((S_q, H, nb), dtype=torch.uint8)
    kv = torch.zeros((S_kv, nb), dtype=torch.uint8)
    qs = torch.full((S_q, H), ONE, dtype=torch.int32)
    ks = torch.full((S_kv,), ONE, dtype=torch.int32)
    w = torch.zeros((S_q, H))
    starts = torch.zeros(S_q, dtype=torch.int32)
    ends = torch.arange(S_q, dtype=torch.int32) + S_kv - S_q
    out = oracle_mod.mx_mqa_logits(q, qs, kv, ks, w, starts, ends, fp4=fp4)
    valid = np.arange(S_kv)[None, :] < ends.numpy()[:, None]
    assert np.array_equal(np.isneginf(out), ~valid)
    assert np.all(out[valid] == 0.0)


def test_unit_scales_reduce_to_fp8_logits(oracle_mod):
    case = wl.mx_dense_case(24, 200, 8, seed=41, sf_lo=127, sf_hi=127)
    got, gtol = oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                         case.k_start, case.k_end, with_tol=True)
    want, wtol = oracle_mod.mqa_logits(case.q, case.kv, torch.ones(case.S_kv), case.weights,
                                       case.k_start, case.k_end, with_tol=True)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.allclose(gtol, wtol, rtol=1e-12, atol=0)


@pytest.mark.parametrize("fp4", [False, True])
def test_single_head_reduces_to_matmul(oracle_mod, fp4):
    case = wl.mx_dense_case(20, 70, 1, seed=42 + fp4, fp4=fp4, ranges="full")
    case.weights = torch.ones_like(case.weights)
    got = oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                   case.k_start, case.k_end, fp4=fp4)
    qd = decode_scaled(case, "q")[:, 0, :]
    kd = decode_scaled(case, "kv")
    ref = torch.relu(qd @ kd.T).to(torch.float32).numpy()
    assert np.allclose(got, ref, rtol=1e-6, atol=0)


@pytest.mark.parametrize("which,block", [("q", 0), ("q", 3), ("kv", 1), ("kv", 2)])
def test_block_scale_is_a_power_of_two_of_its_block(oracle_mod, which, block):
    case = wl.mx_dense_case(12, 40, 4, seed=43, ranges="full")
    # keep only this block's elements, so its scale alone sets the result
    keep = torch.zeros(128, dtype=torch.bool)
    keep[32 * block:32 * block + 32] = True
    case.q = torch.where(keep, case.q, torch.zeros_like(case.q))
    case.kv = torch.where(keep, case.kv, torch.zeros_like(case.kv))
    base = oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                    case.k_start, case.k_end)
    bump = 1 << (8 * block)
    if which == "q":
        case.q_sf = ((case.q_sf.to(torch.int64) + bump + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32)
    else:
        case.kv_sf = ((case.kv_sf.to(torch.int64) + bump + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32)
    up = oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                  case.k_start, case.k_end)
    assert np.array_equal(up, 2 * base)
    # bumping another block's scale changes nothing
    other = (block + 1) % 4
    if which == "q":
        case.q_sf = (case.q_sf.to(torch.int64) + (1 << (8 * other)))
        case.q_sf = ((case.q_sf + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32)
    else:
        case.kv_sf = (case.kv_sf.to(torch.int64) + (1 << (8 * other)))
        case.kv_sf = ((case.kv_sf + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32)
    same = oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                    case.k_start, case.k_end)
    assert np.array_equal(same, up)


def test_hand_derived_block_cases(oracle_mod):
    one = torch.tensor(1.0).to(torch.float8_e4m3fn).view(torch.uint8).item()
    # H = 1, one key; q and kv are 1.0 in block 2 only; byte 2 of q's scale is
    # 128 (x2) and byte 2 of kv's is 126 (x0.5), the rest 127:
    # x = 32 * (1 * 2) * (1 * 0.5) = 32, weight 3 -> 96
    q = torch.zeros((1, 1, 128), dtype=torch.uint8)
    kv = torch.zeros((1, 128), dtype=torch.uint8)
    q[0, 0, 64:96] = one
    kv[0, 64:96] = one
    qs = torch.tensor([[sf(127, 127, 128, 127)]], dtype=torch.int32)
    ks = torch.tensor([sf(127, 127, 126, 127)], dtype=torch.int32)
    w = torch.tensor([[3.0]])
    r = lambda qs_, ks_, w_: oracle_mod.mx_mqa_logits(q, qs_, kv, ks_, w_, torch.tensor([0], dtype=torch.int32),
                                                    torch.tensor([1], dtype=torch.int32))[0, 0]
    assert r(qs, ks, w) == 96.0
    # the same scales on byte 1 leave block 2 at scale one: x = 32 -> 96
    assert r(torch.tensor([[sf(127, 128, 127, 127)]], dtype=torch.int32),
             torch.tensor([sf(127, 126, 127, 127)], dtype=torch.int32), w) == 96.0
    assert r(torch.tensor([[sf(127, 128, 127, 127)]], dtype=torch.int32), ks, w) == 48.0
    # a negative weight on a positive x, and a negative x under the ReLU
    assert r(qs, ks, torch.tensor([[-3.0]])) == -96.0
    kv[0, 64:96] = torch.tensor(-1.0).to(torch.float8_e4m3fn).view(torch.uint8).item()
    assert r(qs, ks, w) == 0.0


def test_e2m1_hand_case(oracle_mod):
    # byte 0x21 holds codes 1 and 2 (0.5 and 1.0), byte 0x3E codes 14 and 3
    # (-4.0 and 1.5); against kv codes 2 (1.0) everywhere in block 0:
    # x = 0.5 + 1.0 - 4.0 + 1.5 = -1.0 -> ReLU 0; with kv code 10 (-1.0): x = 1.0
    q = torch.zeros((1, 1, 64), dtype=torch.uint8)
    q[0, 0, 0], q[0, 0, 1] = 0x21, 0x3E
    kv = torch.zeros((2, 64), dtype=torch.uint8)
    kv[0, :16] = 0x22
    kv[1, :16] = 0xAA
    one = torch.tensor([[ONE]], dtype=torch.int32)
    out = oracle_mod.mx_mqa_logits(q, one, kv, torch.tensor([ONE, ONE], dtype=torch.int32),
                                   torch.tensor([[2.0]]), torch.tensor([0], dtype=torch.int32),
                                   torch.tensor([2], dtype=torch.int32), fp4=True)
    assert out[0].tolist() == [0.0, 2.0]


def test_nibble_order_is_unobservable(oracle_mod):
    # swapping the two nibbles of every byte of q and kv alike permutes the
    # elements within each block, so no logit changes
    case = wl.mx_dense_case(10, 50, 4, seed=44, fp4=True, ranges="full")
    a = oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                 case.k_start, case.k_end, fp4=True)
    swap = lambda t: ((t >> 4) | ((t & 0xF) << 4)).to(torch.uint8)
    b = oracle_mod.mx_mqa_logits(swap(case.q), case.q_sf, swap(case.kv), case.kv_sf, case.weights,
                                 case.k_start, case.k_end, fp4=True)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_nonnegative_weights_give_nonnegative_logits(oracle_mod):
    case = wl.mx_dense_case(16, 80, 8, seed=45)
    case.weights = case.weights.abs()
    out = oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                   case.k_start, case.k_end)
    assert np.all(out[np.isfinite(out)] >= 0)


def test_invalid_arguments(oracle_mod):
    case = wl.mx_dense_case(4, 16, 2, seed=46)
    with pytest.raises(ValueError):   # uncompressed rows need ldo >= S_kv
        oracle_mod.mx_mqa_logits(case.q, case.q_sf, case.kv, case.kv_sf, case.weights,
                                 case.k_start, case.k_end, ldo=8)
    with pytest.raises(ValueError):   # D must be 128
        oracle_mod.mx_mqa_logits(case.q[:, :, :64], case.q_sf, case.kv[:, :64], case.kv_sf,
                                 case.weights, case.k_start, case.k_end)


# ------------------------------------------------------------- paged MX
# The paged MX oracle is pinned to the dense MX oracle above by gathering each
# sequence's keys through its block table with plain tensor indexing, and to
# the paged FP8 oracle by unit scales.

def gather_dense(case, b):
    """Keys and scales of sequence b in position order (torch indexing)."""
    n = int((case.block_table[b] >= 0).sum())
    blocks = case.block_table[b, :n].long()
    kv = case.kv_cache[blocks].reshape(n * case.block_kv, case.kv_cache.shape[2])
    ks = case.kv_sf[blocks].reshape(n * case.block_kv)
    return kv, ks


@pytest.mark.parametrize("fp4,next_n,block_kv", [(False, 2, 64), (True, 3, 32), (False, 1, 128)])
def test_paged_mx_equals_dense_mx_of_the_gathered_keys(oracle_mod, fp4, next_n, block_kv):
    ctx = [1, 70, 129, 0, 200]
    case = wl.paged_mx_case(5, next_n, 8, seed=48 + next_n, context_lens=ctx, block_kv=block_kv,
                            fp4=fp4)
    got = oracle_mod.paged_mx_mqa_logits(case.q, case.q_sf, case.kv_cache, case.kv_sf,
                                         case.weights, case.context_lens, case.block_table,
                                         next_n=next_n, fp4=fp4)
    width = case.ldo
    for b, c in enumerate(ctx):
        kv, ks = gather_dense(case, b)
        rows = slice(b * next_n, (b + 1) * next_n)
        t = torch.arange(next_n, dtype=torch.int32)
        ends = (c - next_n + t + 1).clamp(min=0)
        want = oracle_mod.mx_mqa_logits(case.q[rows], case.q_sf[rows], kv, ks, case.weights[rows],
                                        torch.zeros(next_n, dtype=torch.int32), ends, fp4=fp4,
                                        ldo=max(kv.shape[0], 1)) if kv.shape[0] else None
        g = got[rows]
        for i in range(next_n):
            e = int(ends[i])
            assert np.isneginf(g[i, e:]).all()
            if e:
                assert np.array_equal(g[i, :e].view(np.uint32), want[i, :e].view(np.uint32))
        assert g.shape[1] == width


def test_paged_mx_unit_scales_equal_paged_fp8(oracle_mod):
    ctx = [90, 3, 257]
    case = wl.paged_mx_case(3, 2, 16, seed=52, context_lens=ctx, block_kv=64, sf_lo=127, sf_hi=127)
    a = oracle_mod.paged_mx_mqa_logits(case.q, case.q_sf, case.kv_cache, case.kv_sf, case.weights,
                                       case.context_lens, case.block_table, next_n=2)
    ones = torch.ones(case.kv_sf.shape, dtype=torch.float32)
    b = oracle_mod.paged_mqa_logits(case.q, case.kv_cache, ones, case.weights, case.context_lens,
                                    case.block_table, next_n=2)
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = np.isfinite(b)
    assert np.allclose(a[fin], b[fin], rtol=1e-6, atol=1e-6)


def test_paged_mx_hand_case(oracle_mod):
    # one sequence of 3 keys in block 1 (block 0 unused), one head, E2M1 code
    # 2 (1.0) in all 128 elements of q and of key 1; key 2's block 3 scale is
    # 2^1: x = 4 blocks x 32 = 128 for key 1, 3 x 32 + 64 = 160 for key 2
    q = torch.full((1, 1, 64), 0x22, dtype=torch.uint8)
    kv = torch.zeros((2, 4, 64), dtype=torch.uint8)
    kv[1, 1], kv[1, 2] = 0x22, 0x22
    ksf = torch.full((2, 4), ONE, dtype=torch.int32)
    ksf[1, 2] = sf(127, 127, 127, 128)
    out = oracle_mod.paged_mx_mqa_logits(q, torch.tensor([[ONE]], dtype=torch.int32), kv, ksf,
                                         torch.tensor([[0.5]]), torch.tensor([3], dtype=torch.int32),
                                         torch.tensor([[1]], dtype=torch.int32), next_n=1, fp4=True)
    assert out[0].tolist() == [0.0, 64.0, 80.0, float("-inf")]
