"""Pins for the CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics fix
by themselves: hand-derived worked examples (tests/golden/hand_cases.json), a
library routine (torch's E4M3 cast, torch.matmul in float64), closed forms for
+-1 and one-hot inputs, the all-zero case of the PR #435 reproducer, exact
metamorphic relations (power-of-two scaling), invariants and brute force.
They are chosen so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from fp8_mqa_indexer_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def e4m3_bytes(values) -> torch.Tensor:
    t = torch.tensor(values, dtype=torch.float32)
    b = t.to(torch.float8_e4m3fn)
    assert torch.equal(b.to(torch.float32), t), "golden input not exactly representable"
    return b.view(torch.uint8)


def decode(u8: torch.Tensor) -> torch.Tensor:
    """Library decode (torch's own float8_e4m3fn cast) into float64."""
    return u8.view(torch.float8_e4m3fn).to(torch.float64)


# ---------------------------------------------------------------- E4M3 decode
def test_e4m3_table_matches_library_cast(oracle_mod):
    tab = oracle_mod.e4m3_table()
    ref = decode(torch.arange(256, dtype=torch.uint8)).numpy()
    nan_o, nan_r = np.isnan(tab), np.isnan(ref)
    assert np.array_equal(nan_o, nan_r)
    assert set(np.nonzero(nan_o)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(tab[~nan_o], ref[~nan_r])
    # signed zeros: code 0x80 is -0.0
    assert math.copysign(1.0, tab[0x80]) == -1.0


def test_e4m3_landmark_codes(oracle_mod):
    # Landmarks of the OCP FP8 E4M3 format (bias 7, 3 mantissa bits, max 448).
    tab = oracle_mod.e4m3_table()
    assert tab[0x38] == 1.0 and tab[0xB8] == -1.0
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0
    assert tab[0x01] == 2.0 ** -9          # smallest subnormal
    assert tab[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert tab[0x08] == 2.0 ** -6          # smallest normal
    assert tab[0x40] == 2.0


# -------------------------------------------------------------- golden cases
def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_hand_cases(oracle_mod, case):
    q = e4m3_bytes(case["q"])
    kv = e4m3_bytes(case["kv"])
    sc = torch.tensor(case["kv_scale"], dtype=torch.float32)
    w = torch.tensor(case["weights"], dtype=torch.float32)
    ks = torch.tensor(case["k_start"], dtype=torch.int32)
    ke = torch.tensor(case["k_end"], dtype=torch.int32)
    out, tol = oracle_mod.mqa_logits(q, kv, sc, w, ks, ke, ldo=case["ldo"], clean=case["clean"],
                                     compressed=case["compressed"], with_tol=True)
    exp = np.array([[float(v) for v in row] for row in case["expected"]], np.float32)
    assert np.array_equal(out, exp), (out, exp)
    exp_tol = np.array(case["expected_tol"], np.float64)
    assert np.allclose(tol, exp_tol, rtol=1e-12, atol=1e-15), (tol, exp_tol)


# ---------------------------------------------------------- closed forms
def test_pm1_closed_form(oracle_mod):
    """q, kv in {-1,+1}: <q,kv> = D - 2 * (#positions where the signs differ)."""
    g = torch.Generator().manual_seed(7)
    S_q, S_kv, D = 9, 13, 64
    qs = torch.randint(0, 2, (S_q, 1, D), generator=g) * 2 - 1
    ks = torch.randint(0, 2, (S_kv, D), generator=g) * 2 - 1
    q, kv = e4m3_bytes(qs.float().tolist()), e4m3_bytes(ks.float().tolist())
    ones_s = torch.ones(S_kv)
    ones_w = torch.ones(S_q, 1)
    z = torch.zeros(S_q, dtype=torch.int32)
    e = torch.full((S_q,), S_kv, dtype=torch.int32)
    out = oracle_mod.mqa_logits(q, kv, ones_s, ones_w, z, e)
    for i in range(S_q):
        for j in range(S_kv):
            mism = int((qs[i, 0] != ks[j]).sum())
            assert out[i, j] == max(0, D - 2 * mism)


def test_one_hot_single_product(oracle_mod):
    """One-hot rows: the dot product is a single product or exactly zero."""
    S_q, S_kv, D = 6, 7, 16
    qv = np.zeros((S_q, 1, D), np.float32)
    kvv = np.zeros((S_kv, D), np.float32)
    qpos = [(3 * i) % D for i in range(S_q)]
    kpos = [(5 * j) % D for j in range(S_kv)]
    for i in range(S_q):
        qv[i, 0, qpos[i]] = 1.5 + i          # 1.5 .. 6.5, all exact in E4M3
    for j in range(S_kv):
        kvv[j, kpos[j]] = 0.25 * (j + 1)     # 0.25 .. 1.75
    out = oracle_mod.mqa_logits(e4m3_bytes(qv.tolist()), e4m3_bytes(kvv.tolist()),
                                torch.ones(S_kv), torch.ones(S_q, 1),
                                torch.zeros(S_q, dtype=torch.int32),
                                torch.full((S_q,), S_kv, dtype=torch.int32))
    for i in range(S_q):
        for j in range(S_kv):
            want = (1.5 + i) * 0.25 * (j + 1) if qpos[i] == kpos[j] else 0.0
            assert out[i, j] == np.float32(want)


def test_all_zero_inputs_give_zero_and_neg_inf(oracle_mod):
    """PR #435 reproducer: zero Q/K/W -> exactly 0 inside ranges, -inf outside."""
    S_q, S_kv, H, D = 17, 260, 4, 64
    z8 = torch.zeros((S_q, H, D), dtype=torch.uint8)
    kv = torch.zeros((S_kv, D), dtype=torch.uint8)
    ends = torch.arange(S_q, dtype=torch.int32) + S_kv - S_q
    out = oracle_mod.mqa_logits(z8, kv, torch.ones(S_kv), torch.zeros(S_q, H),
                                torch.zeros(S_q, dtype=torch.int32), ends)
    cols = np.arange(S_kv)[None, :]
    valid = cols < ends.numpy()[:, None]
    assert np.array_equal(np.isneginf(out), ~valid)
    assert (out[valid] == 0).all()


def test_single_head_reduces_to_matmul(oracle_mod):
    """H=1, w=1, s=1, full ranges: logits = relu(Q @ KV^T), with torch.matmul in
    float64 on library-decoded values (exact for E4M3 inputs at this D)."""
    case = wl.dense_case(37, 300, 1, 128, seed=11, ranges="full")
    s1 = torch.ones(case.S_kv)
    w1 = torch.ones(case.S_q, 1)
    out = oracle_mod.mqa_logits(case.q, case.kv, s1, w1, case.k_start, case.k_end)
    ref = torch.relu(decode(case.q[:, 0, :]) @ decode(case.kv).T).to(torch.float32).numpy()
    assert np.array_equal(out, ref)


def test_head_selection_by_one_hot_weights(oracle_mod):
    """With w = e_h the multi-head logit equals the single-head logit of head h
    (catches a head/dim transpose or a wrong head index)."""
    case = wl.dense_case(5, 40, 4, 64, seed=12, ranges="full")
    for h in range(4):
        w = torch.zeros(case.S_q, 4)
        w[:, h] = 1.0
        multi = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, w, case.k_start, case.k_end)
        single = oracle_mod.mqa_logits(case.q[:, h:h + 1, :].contiguous(), case.kv, case.kv_scale,
                                       torch.ones(case.S_q, 1), case.k_start, case.k_end)
        assert np.array_equal(multi, single)


def test_single_head_with_scale_matches_matmul(oracle_mod):
    """H=1, w=1: logits = relu(s_j * (Q @ KV^T)[i, j]) by torch, per column scale."""
    case = wl.dense_case(23, 129, 1, 64, seed=13, ranges="full")
    out = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, torch.ones(case.S_q, 1),
                                case.k_start, case.k_end)
    x = decode(case.q[:, 0, :]) @ decode(case.kv).T
    ref = torch.relu(x * case.kv_scale.to(torch.float64)[None, :]).to(torch.float32).numpy()
    assert np.array_equal(out, ref)


# ------------------------------------------------------- metamorphic / invariants
def test_power_of_two_scaling_is_exact(oracle_mod):
    case = wl.dense_case(19, 150, 8, 64, seed=14, ranges="causal_tail_inclusive")
    base = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start, case.k_end)
    s2 = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale * 2, case.weights, case.k_start, case.k_end)
    w2 = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights * 4, case.k_start, case.k_end)
    fin = np.isfinite(base)
    assert np.array_equal(np.isneginf(base), np.isneginf(s2))
    assert np.array_equal(s2[fin], 2 * base[fin])
    assert np.array_equal(w2[fin], 4 * base[fin])


def test_weight_linearity(oracle_mod):
    case = wl.dense_case(11, 70, 8, 64, seed=15, ranges="full")
    w_a = case.weights
    w_b = torch.randn(case.weights.shape, generator=torch.Generator().manual_seed(3))
    f = lambda w: oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, w, case.k_start,
                                        case.k_end).astype(np.float64)
    lhs = f(w_a + w_b)
    rhs = f(w_a) + f(w_b)
    scale = f(w_a.abs()) + f(w_b.abs()) + 1e-30
    assert np.all(np.abs(lhs - rhs) <= 4e-7 * scale + 1e-30)


def test_nonnegative_weights_give_nonnegative_logits(oracle_mod):
    case = wl.dense_case(21, 200, 8, 64, seed=16, ranges="suffix")
    out = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights.abs(),
                                case.k_start, case.k_end)
    fin = np.isfinite(out)
    assert (out[fin] >= 0).all()
    # -inf count = sum over rows of (width - range length)
    assert int(np.isneginf(out).sum()) == int((case.S_kv - case.valid_counts()).sum())


def test_key_permutation_permutes_columns(oracle_mod):
    case = wl.dense_case(7, 50, 4, 64, seed=17, ranges="full")
    perm = torch.randperm(case.S_kv, generator=torch.Generator().manual_seed(5))
    a = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start, case.k_end)
    b = oracle_mod.mqa_logits(case.q, case.kv[perm].contiguous(), case.kv_scale[perm].contiguous(),
                              case.weights, case.k_start, case.k_end)
    assert np.array_equal(b, a[:, perm.numpy()])


def test_nonclean_leaves_outside_untouched(oracle_mod):
    case = wl.dense_case(9, 64, 4, 64, seed=18, ranges="suffix")
    sentinel = np.full((case.S_q, case.S_kv), 12345.0, np.float32)
    out = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                case.k_end, clean=False, out=sentinel)
    clean = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start, case.k_end)
    inside = np.isfinite(clean)
    assert np.array_equal(out[inside], clean[inside])
    assert (out[~inside] == 12345.0).all()


def test_compressed_is_shifted_uncompressed(oracle_mod):
    case = wl.dense_case(13, 90, 4, 64, seed=19, ranges="custom",
                         k_start=[3 * i for i in range(13)], k_end=[40 + 3 * i for i in range(13)])
    full = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start, case.k_end)
    comp = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                                 case.k_end, ldo=45, compressed=True)
    for i in range(13):
        lo, hi = 3 * i, min(40 + 3 * i, 90)
        assert np.array_equal(comp[i, :hi - lo], full[i, lo:hi])
        assert np.isneginf(comp[i, hi - lo:]).all()


def test_ranges_clip_to_existing_keys(oracle_mod):
    case = wl.dense_case(4, 30, 2, 64, seed=20, ranges="custom", k_start=[-5, 10, 25, 7],
                         k_end=[12, 50, 20, 7])
    out = oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start, case.k_end)
    assert np.isfinite(out[0, :12]).all() and np.isneginf(out[0, 12:]).all()
    assert np.isneginf(out[1, :10]).all() and np.isfinite(out[1, 10:]).all()
    assert np.isneginf(out[2]).all() and np.isneginf(out[3]).all()


def test_invalid_arguments_rejected(oracle_mod):
    case = wl.dense_case(4, 30, 2, 64, seed=21, ranges="full")
    with pytest.raises(ValueError):
        oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                              case.k_end, ldo=10)
    with pytest.raises(ValueError):   # compressed row longer than ldo
        oracle_mod.mqa_logits(case.q, case.kv, case.kv_scale, case.weights, case.k_start,
                              case.k_end, ldo=10, compressed=True)


# ------------------------------------------------------------------- paged
def _small_paged(seed=30, B=5, next_n=2, block_kv=64, ctx=None):
    return wl.paged_case(B, next_n, 4, 64, seed=seed, ctx_lo=1, ctx_hi=700, block_kv=block_kv,
                         num_blocks=80, context_lens=ctx)


@pytest.mark.parametrize("next_n,block_kv", [(1, 64), (2, 64), (3, 32), (4, 64)])
def test_paged_equals_dense_on_gathered_keys(oracle_mod, next_n, block_kv):
    case = _small_paged(next_n=next_n, block_kv=block_kv,
                        ctx=[1, 700, 64, 129, next_n - 1 if next_n > 1 else 0])
    paged = oracle_mod.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, case.weights,
                                        case.context_lens, case.block_table, next_n=next_n)
    width = case.max_blocks_per_seq * case.block_kv
    for b in range(case.B):
        ctx = int(case.context_lens[b])
        n_pages = (ctx + block_kv - 1) // block_kv
        ids = case.block_table[b, :n_pages].long()
        kv = case.kv_cache[ids].reshape(-1, case.D)[:ctx].contiguous()
        sc = case.kv_scales[ids].reshape(-1)[:ctx].contiguous()
        if ctx == 0:
            kv = torch.zeros((1, case.D), dtype=torch.uint8)
            sc = torch.ones(1)
        rows = slice(b * next_n, (b + 1) * next_n)
        t = torch.arange(next_n, dtype=torch.int32)
        ends = (ctx - next_n + t + 1).clamp(min=0)
        dense = oracle_mod.mqa_logits(case.q[rows].contiguous(), kv, sc, case.weights[rows].contiguous(),
                                      torch.zeros(next_n, dtype=torch.int32), ends.to(torch.int32),
                                      ldo=width)
        got = paged[rows]
        n = kv.shape[0]
        assert np.array_equal(got[:, :n], dense[:, :n])
        assert np.isneginf(got[:, max(ctx, 0):]).all()


def test_paged_rejects_bad_block_ids(oracle_mod):
    case = _small_paged()
    bt = case.block_table.clone()
    bt[1, 0] = case.num_blocks   # out of range
    with pytest.raises(ValueError):
        oracle_mod.paged_mqa_logits(case.q, case.kv_cache, case.kv_scales, case.weights,
                                    case.context_lens, bt, next_n=2)


def _brute_force_schedule(ctx, num_sms):
    units = []
    for b, c in enumerate(ctx):
        for t in range((max(c, 0) + 127) // 128):
            units.append((b, t))
    U = len(units)
    out = []
    for k in range(num_sms + 1):
        u = k * U // num_sms
        out.append(units[u] if u < U else (len(ctx), 0))
    return np.array(out, np.int32), units


@pytest.mark.parametrize("ctx,num_sms", [
    ([1, 700, 64, 129, 0], 4), ([4096, 65536, 5000], 152), ([0, 0, 0], 3),
    ([128] * 10, 10), ([300], 1), (list(range(0, 3000, 97)), 7)])
def test_metadata_brute_force(oracle_mod, ctx, num_sms):
    meta = oracle_mod.paged_mqa_logits_metadata(np.array(ctx, np.int32), next_n=2, block_kv=64,
                                                num_sms=num_sms)
    want, units = _brute_force_schedule(ctx, num_sms)
    assert np.array_equal(meta, want)
    # invariants: monotone, every unit exactly once, chunk sizes differ by at most one
    idx = [units.index(tuple(e)) if tuple(e) in units else len(units) for e in meta.tolist()]
    assert idx == sorted(idx) and idx[0] == 0 and idx[-1] == len(units)
    sizes = np.diff(idx)
    assert sizes.max() - sizes.min() <= 1 if len(sizes) else True


def _brute_force_dense_schedule(k_start, k_end, S_kv, H, num_sms):
    """Units listed from the validity mask itself: block b covers every 128-key
    tile between the tile of its first valid key and the tile of its last."""
    tok = 256 // H
    S_q = len(k_start)
    cols = np.arange(S_kv)
    units = []
    for b in range(0, -(-S_q // tok)):
        rows = range(b * tok, min(S_q, (b + 1) * tok))
        valid = np.zeros(S_kv, bool)
        for i in rows:
            valid |= (cols >= k_start[i]) & (cols < k_end[i])
        keys = np.nonzero(valid)[0]
        if len(keys):
            for t in range(keys[0] // 128, keys[-1] // 128 + 1):
                units.append((b, t))
    U = len(units)
    nb = -(-S_q // tok)
    return np.array([units[k * U // num_sms] if k * U // num_sms < U else (nb, 0)
                     for k in range(num_sms + 1)], np.int32), units


@pytest.mark.parametrize("S_q,S_kv,H,kind,num_sms", [
    (128, 512, 8, "causal", 4), (2048, 4096, 32, "suffix", 152), (300, 1000, 64, "random", 7),
    (17, 260, 64, "random", 152), (64, 300, 64, "empty", 5), (256, 2048, 64, "windows", 13),
    (5, 129, 8, "random", 1)])
def test_dense_metadata_brute_force(oracle_mod, S_q, S_kv, H, kind, num_sms):
    g = np.random.default_rng(S_q + S_kv + H)
    i = np.arange(S_q)
    if kind == "causal":
        ks, ke = np.zeros(S_q), S_kv - S_q + i + 1
    elif kind == "suffix":
        ks, ke = i, np.full(S_q, S_kv)
    elif kind == "empty":
        ks, ke = np.full(S_q, 10), np.full(S_q, 10)
        ke[S_q // 2] = 300                    # one non-empty row
    elif kind == "windows":
        ks = g.integers(0, S_kv, S_q)
        ke = ks + g.integers(0, 300, S_q)     # may run past S_kv (clipped)
    else:
        ks = g.integers(-50, S_kv, S_q)
        ke = g.integers(-50, S_kv + 50, S_q)  # inverted, negative and clipped ranges
    ks, ke = ks.astype(np.int32), ke.astype(np.int32)
    meta = oracle_mod.mqa_logits_metadata(ks, ke, S_kv=S_kv, H=H, num_sms=num_sms)
    want, units = _brute_force_dense_schedule(ks, ke, S_kv, H, num_sms)
    assert np.array_equal(meta, want)
    idx = [units.index(tuple(e)) if tuple(e) in units else len(units) for e in meta.tolist()]
    assert idx == sorted(idx) and idx[0] == 0 and idx[-1] == len(units)


def test_dense_metadata_rejects_invalid_arguments(oracle_mod):
    z = np.zeros(4, np.int32)
    for kw in (dict(S_kv=-1, H=64, num_sms=4), dict(S_kv=10, H=48, num_sms=4),
               dict(S_kv=10, H=64, num_sms=0)):
        with pytest.raises(ValueError):
            oracle_mod.mqa_logits_metadata(z, z, **kw)
