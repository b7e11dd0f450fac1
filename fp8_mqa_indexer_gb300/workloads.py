"""Seeded synthetic inputs for MQA logits scoring.

This module only draws random numbers and lays them out: it holds none of the
scoring arithmetic, and both the CUDA path and the CPU oracle are fed from it.
Every tensor is created on the CPU from a seeded ``torch.Generator`` so the
oracle and the GPU see identical bytes.  FP8 values are produced with torch's
own ``float8_e4m3fn`` cast (round to nearest even) and handed over as raw bytes.

The shapes and distributions follow the workloads the pages describe:
  * the dense call of the instagit DeepGEMM article, section "Implementing
    Standard MQA Logits Computation" (S_q=2048, S_kv=4096, H=32, D=64, ranges
    [i, S_kv));
  * the H=64 / D=128 timing shapes of "[PR #435] Improve SM100 MX MQA logits
    clean-output performance", section "Performance" (Q/KV 2048/32768 and
    8192/65536, each row using [0, KV - Q + row));
  * paged decode as in the article's "Implementing Paged MQA Logits Computation
    for Decoding" with next_n and 64-token blocks as in "[PR #314] fix: SM90
    paged MQA logits IMA on next_n=4";
  * logits-shaped rows for the top-k key selection (N(0,1) values, -inf
    outside each row's range), sized like the 2048 x 32768 dense output;
  * MX inputs (E4M3 or packed E2M1 elements, UE8M0 block scales packed four
    to an int32) with the shapes of the PR #435 reproducer.
The datasets behind those numbers are not public inputs; these synthetic
tensors stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

E4M3 = torch.float8_e4m3fn


@dataclass
class DenseCase:
    name: str
    q: torch.Tensor          # [S_q, H, D] uint8 (E4M3 bytes)
    kv: torch.Tensor         # [S_kv, D] uint8 (E4M3 bytes)
    kv_scale: torch.Tensor   # [S_kv] float32
    weights: torch.Tensor    # [S_q, H] float32
    k_start: torch.Tensor    # [S_q] int32
    k_end: torch.Tensor      # [S_q] int32
    ldo: int
    clean: bool = True
    compressed: bool = False

    @property
    def S_q(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def S_kv(self):
        return self.kv.shape[0]

    def valid_counts(self) -> torch.Tensor:
        """Number of scored keys per row (range clipped to [0, S_kv))."""
        lo = self.k_start.clamp(min=0).to(torch.int64)
        hi = self.k_end.clamp(max=self.S_kv).to(torch.int64)
        return (hi - lo).clamp(min=0)


@dataclass
class PagedCase:
    name: str
    q: torch.Tensor            # [B*next_n, H, D] uint8
    kv_cache: torch.Tensor     # [num_blocks, block_kv, D] uint8
    kv_scales: torch.Tensor    # [num_blocks, block_kv] float32
    weights: torch.Tensor      # [B*next_n, H] float32
    context_lens: torch.Tensor  # [B] int32
    block_table: torch.Tensor  # [B, max_blocks_per_seq] int32 (-1 = unused)
    next_n: int
    ldo: int
    clean: bool = True

    @property
    def B(self):
        return self.context_lens.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def block_kv(self):
        return self.kv_cache.shape[1]

    @property
    def num_blocks(self):
        return self.kv_cache.shape[0]

    @property
    def max_blocks_per_seq(self):
        return self.block_table.shape[1]

    def valid_counts(self) -> torch.Tensor:
        ctx = self.context_lens.to(torch.int64).repeat_interleave(self.next_n)
        t = torch.arange(self.next_n, dtype=torch.int64).repeat(self.B)
        return (ctx - self.next_n + t + 1).clamp(min=0)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def e4m3_normal(shape, g: torch.Generator, clamp: Optional[float] = None,
                chunk: int = 1 << 24) -> torch.Tensor:
    """E4M3 bytes of N(0,1) samples (optionally clamped), drawn in chunks."""
    n = 1
    for s in shape:
        n *= s
    out = torch.empty(n, dtype=torch.uint8)
    for k in range(0, n, chunk):
        m = min(chunk, n - k)
        x = torch.randn(m, generator=g)
        if clamp is not None:
            x = x.clamp(-clamp, clamp)
        out[k:k + m] = x.to(E4M3).view(torch.uint8)
    return out.view(*shape)


def uniform(shape, lo: float, hi: float, g: torch.Generator) -> torch.Tensor:
    return torch.rand(shape, generator=g) * (hi - lo) + lo


def dense_case(S_q: int, S_kv: int, H: int, D: int, *, seed: int, ranges: str = "causal_tail",
               w_std: float = 1.0, clamp: Optional[float] = None, name: str = "dense",
               compressed: bool = False, clean: bool = True, ldo: Optional[int] = None,
               k_start=None, k_end=None) -> DenseCase:
    """A dense case with one of the pages' range shapes.

    ranges: "causal_tail" -> [0, S_kv - S_q + i)       (reproducer of PR #435)
            "causal_tail_inclusive" -> [0, S_kv - S_q + i + 1)
            "suffix" -> [i, S_kv)                        (instagit dense example)
            "full" -> [0, S_kv)
            "custom" -> k_start / k_end given
    """
    g = _gen(seed)
    q = e4m3_normal((S_q, H, D), g, clamp)
    kv = e4m3_normal((S_kv, D), g, clamp)
    kv_scale = uniform((S_kv,), 0.5, 2.0, g)
    weights = torch.randn((S_q, H), generator=g) * w_std
    i = torch.arange(S_q, dtype=torch.int32)
    if ranges == "causal_tail":
        ks, ke = torch.zeros_like(i), S_kv - S_q + i
    elif ranges == "causal_tail_inclusive":
        ks, ke = torch.zeros_like(i), S_kv - S_q + i + 1
    elif ranges == "suffix":
        ks, ke = i.clone(), torch.full_like(i, S_kv)
    elif ranges == "full":
        ks, ke = torch.zeros_like(i), torch.full_like(i, S_kv)
    elif ranges == "custom":
        ks = torch.as_tensor(k_start, dtype=torch.int32)
        ke = torch.as_tensor(k_end, dtype=torch.int32)
    else:
        raise ValueError(ranges)
    ks, ke = ks.to(torch.int32).contiguous(), ke.to(torch.int32).contiguous()
    if ldo is None:
        if compressed:
            lens = (ke.clamp(max=S_kv) - ks.clamp(min=0)).clamp(min=0)
            ldo = max(1, int(lens.max().item()) if S_q else 1)
        else:
            ldo = S_kv
    return DenseCase(name, q, kv, kv_scale, weights, ks, ke, ldo, clean, compressed)


# Named workloads.  Index order is the order the benchmark configuration lists them.
DENSE_CONFIGS = {
    "dense_tiny": dict(S_q=128, S_kv=512, H=8, D=64, ranges="causal_tail_inclusive", clamp=4.0,
                       seed=1000),
    "dense_2k_4k_h32_d64": dict(S_q=2048, S_kv=4096, H=32, D=64, ranges="suffix", seed=1001),
    "dense_2k_32k_h64_d128": dict(S_q=2048, S_kv=32768, H=64, D=128, ranges="causal_tail",
                                  w_std=0.125, seed=1002),
    "dense_8k_64k_h64_d128": dict(S_q=8192, S_kv=65536, H=64, D=128, ranges="causal_tail",
                                  w_std=0.125, seed=1003),
    "dense_8k_64k_h64_d128_compressed": dict(S_q=8192, S_kv=65536, H=64, D=128,
                                             ranges="causal_tail", w_std=0.125, seed=1003,
                                             compressed=True),
}


def dense_config(name: str) -> DenseCase:
    return dense_case(name=name, **DENSE_CONFIGS[name])


def paged_case(B: int, next_n: int, H: int, D: int, *, seed: int, ctx_lo: int, ctx_hi: int,
               block_kv: int = 64, num_blocks: int = 70000, max_blocks_per_seq: Optional[int] = None,
               name: str = "paged", context_lens=None) -> PagedCase:
    """Paged decode case: random context lengths in [ctx_lo, ctx_hi], pages of
    ``block_kv`` keys handed out by a random permutation of the physical blocks."""
    g = _gen(seed)
    if context_lens is None:
        ctx = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=g, dtype=torch.int64)
    else:
        ctx = torch.as_tensor(context_lens, dtype=torch.int64)
    pages = (ctx.clamp(min=0) + block_kv - 1) // block_kv
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, (ctx_hi + block_kv - 1) // block_kv)
    assert int(pages.sum()) <= num_blocks and int(pages.max()) <= max_blocks_per_seq
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    table = torch.full((B, max_blocks_per_seq), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(pages[b])
        table[b, :n] = perm[off:off + n]
        off += n
    kv_cache = e4m3_normal((num_blocks, block_kv, D), g)
    kv_scales = uniform((num_blocks, block_kv), 0.5, 2.0, g)
    q = e4m3_normal((B * next_n, H, D), g)
    weights = torch.randn((B * next_n, H), generator=g)
    ldo = max_blocks_per_seq * block_kv
    return PagedCase(name, q, kv_cache, kv_scales, weights, ctx.to(torch.int32), table, next_n, ldo)


PAGED_CONFIGS = {
    "paged_b64_n2_h64_d128": dict(B=64, next_n=2, H=64, D=128, ctx_lo=4096, ctx_hi=65536,
                                  block_kv=64, num_blocks=70000, seed=1004),
}


def paged_config(name: str) -> PagedCase:
    return paged_case(name=name, **PAGED_CONFIGS[name])


@dataclass
class TopkCase:
    """Input of the top-k key selection: a logits matrix and its row ranges."""
    name: str
    logits: torch.Tensor    # [rows, ldo] float32
    k_start: torch.Tensor   # [rows] int32
    k_end: torch.Tensor     # [rows] int32
    n_cols: int             # keys of an uncompressed row
    topk: int
    compressed: bool = False

    @property
    def rows(self):
        return self.logits.shape[0]

    @property
    def ldo(self):
        return self.logits.shape[1]

    def valid_counts(self) -> torch.Tensor:
        lo = self.k_start.to(torch.int64).clamp(0, self.n_cols)
        hi = self.k_end.to(torch.int64).clamp(max=self.n_cols)
        n = (hi - lo).clamp(min=0)
        return n.clamp(max=self.ldo) if self.compressed else n


def topk_case(rows: int, n_cols: int, topk: int, *, seed: int, ranges: str = "causal_tail",
              levels: int = 0, ldo: Optional[int] = None, name: str = "topk",
              k_start=None, k_end=None) -> TopkCase:
    """Logits-shaped rows for the top-k selection: N(0,1) fp32 values (rounded
    to multiples of 1/levels when ``levels`` > 0, which makes exact ties common)
    and -inf outside each row's range, as clean logits have.  ``ranges`` as in
    ``dense_case`` with S_q = rows and S_kv = n_cols."""
    g = _gen(seed)
    L = torch.empty((rows, ldo or n_cols), dtype=torch.float32)
    chunk = max(1, (1 << 24) // max(1, L.shape[1]))
    for r in range(0, rows, chunk):
        x = torch.randn((min(chunk, rows - r), L.shape[1]), generator=g)
        if levels:
            x = torch.round(x * levels) / levels
        L[r:r + x.shape[0]] = x
    i = torch.arange(rows, dtype=torch.int32)
    if ranges == "causal_tail":
        ks, ke = torch.zeros_like(i), n_cols - rows + i
    elif ranges == "full":
        ks, ke = torch.zeros_like(i), torch.full_like(i, n_cols)
    elif ranges == "custom":
        ks = torch.as_tensor(k_start, dtype=torch.int32)
        ke = torch.as_tensor(k_end, dtype=torch.int32)
    else:
        raise ValueError(ranges)
    cols = torch.arange(L.shape[1], dtype=torch.int64)[None, :]
    outside = (cols < ks.to(torch.int64)[:, None]) | (cols >= ke.to(torch.int64)[:, None])
    L[outside] = float("-inf")
    return TopkCase(name, L, ks.contiguous(), ke.contiguous(), n_cols, topk)


# The selection over rows shaped like the 2048 x 32768 dense workload's logits,
# k = 2048 (the pages leave k to the caller).
TOPK_CONFIGS = {
    "topk_2k_32k_k2048": dict(rows=2048, n_cols=32768, topk=2048, ranges="causal_tail", seed=1005),
}


def topk_config(name: str) -> TopkCase:
    return topk_case(name=name, **TOPK_CONFIGS[name])


# Fused logits + top-k: the dense workload's inputs (non-clean, the fused call
# writes no logits) and the number of keys kept per row.
FUSED_CONFIGS = {
    "fused_topk_2k_32k_h64_d128_k2048": dict(dense="dense_2k_32k_h64_d128", topk=2048),
    "fused_topk_8k_64k_h64_d128_k2048": dict(dense="dense_8k_64k_h64_d128", topk=2048),
}


def fused_config(name: str):
    """(dense case, topk) of a fused logits + top-k workload."""
    cfg = FUSED_CONFIGS[name]
    case = dense_config(cfg["dense"])
    case.name = name
    case.clean = False
    return case, cfg["topk"]


@dataclass
class MxDenseCase:
    """Dense MX (block-scaled) input: E4M3 or packed E2M1 elements with four
    UE8M0 block scales per 128-element row, packed in an int32."""
    name: str
    q: torch.Tensor          # [S_q, H, 128] uint8 (E4M3) or [S_q, H, 64] uint8 (E2M1 pairs)
    q_sf: torch.Tensor       # [S_q, H] int32
    kv: torch.Tensor         # [S_kv, 128] or [S_kv, 64] uint8
    kv_sf: torch.Tensor      # [S_kv] int32
    weights: torch.Tensor    # [S_q, H] float32
    k_start: torch.Tensor    # [S_q] int32
    k_end: torch.Tensor      # [S_q] int32
    fp4: bool
    ldo: int

    @property
    def S_q(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def S_kv(self):
        return self.kv.shape[0]

    D = 128
    clean = True
    compressed = False

    def valid_counts(self) -> torch.Tensor:
        """Number of scored keys per row (range clipped to [0, S_kv))."""
        lo = self.k_start.clamp(min=0).to(torch.int64)
        hi = self.k_end.clamp(max=self.S_kv).to(torch.int64)
        return (hi - lo).clamp(min=0)


def packed_scales(shape, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    """int32 tensor whose four bytes are independent UE8M0 codes in [lo, hi]."""
    b = torch.randint(lo, hi + 1, tuple(shape) + (4,), generator=g, dtype=torch.int64)
    v = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)
    return torch.where(v >= 1 << 31, v - (1 << 32), v).to(torch.int32)


def e2m1_pairs(shape, g: torch.Generator) -> torch.Tensor:
    """Bytes of two uniformly drawn E2M1 codes each (``shape`` in bytes)."""
    lo = torch.randint(0, 16, shape, generator=g, dtype=torch.int64)
    hi = torch.randint(0, 16, shape, generator=g, dtype=torch.int64)
    return (lo | (hi << 4)).to(torch.uint8)


def mx_dense_case(S_q: int, S_kv: int, H: int, *, seed: int, fp4: bool = False,
                  ranges: str = "causal_tail", sf_lo: int = 124, sf_hi: int = 130,
                  name: str = "mx_dense") -> MxDenseCase:
    """MX dense case, D = 128: E4M3 elements from N(0,1) (or uniform E2M1
    codes), block scales drawn uniformly from [sf_lo, sf_hi] (127 is one), the
    dense ranges of ``dense_case``."""
    g = _gen(seed)
    D = 128
    if fp4:
        q, kv = e2m1_pairs((S_q, H, D // 2), g), e2m1_pairs((S_kv, D // 2), g)
    else:
        q, kv = e4m3_normal((S_q, H, D), g), e4m3_normal((S_kv, D), g)
    q_sf = packed_scales((S_q, H), sf_lo, sf_hi, g)
    kv_sf = packed_scales((S_kv,), sf_lo, sf_hi, g)
    weights = torch.randn((S_q, H), generator=g)
    i = torch.arange(S_q, dtype=torch.int32)
    if ranges == "causal_tail":
        ks, ke = torch.zeros_like(i), S_kv - S_q + i
    elif ranges == "full":
        ks, ke = torch.zeros_like(i), torch.full_like(i, S_kv)
    else:
        raise ValueError(ranges)
    return MxDenseCase(name, q, q_sf, kv, kv_sf, weights, ks.contiguous(), ke.contiguous(), fp4, S_kv)


def mx_zero_case(S_q: int, S_kv: int, H: int, *, fp4: bool = False,
                 name: str = "mx_zeros") -> MxDenseCase:
    """The PR #435 reproducer's MX input: all-zero q, k and weights (E4M3, or
    packed E2M1 with 64 bytes per row), every scale byte 127 (0x7f7f7f7f:
    one), rows [0, S_kv - S_q + i)."""
    nb = 64 if fp4 else 128
    i = torch.arange(S_q, dtype=torch.int32)
    one = torch.tensor(0x7F7F7F7F, dtype=torch.int32)
    return MxDenseCase(name, torch.zeros((S_q, H, nb), dtype=torch.uint8),
                       one.repeat(S_q * H).reshape(S_q, H), torch.zeros((S_kv, nb), dtype=torch.uint8),
                       one.repeat(S_kv), torch.zeros((S_q, H)), torch.zeros_like(i),
                       (S_kv - S_q + i).contiguous(), fp4, S_kv)


# The MXFP8 timing shapes of "[PR #435] ...", section "Performance" (seeded
# random elements and scales; "_zeros": the reproducer's all-zero input).
MX_CONFIGS = {
    "mx_2k_32k_h64_d128": dict(S_q=2048, S_kv=32768, H=64, seed=1010),
    "mx_8k_64k_h64_d128": dict(S_q=8192, S_kv=65536, H=64, seed=1011),
    "mx_2k_32k_h64_d128_zeros": dict(S_q=2048, S_kv=32768, H=64, zeros=True),
    "mx_8k_64k_h64_d128_zeros": dict(S_q=8192, S_kv=65536, H=64, zeros=True),
    "mx4_2k_32k_h64_d128": dict(S_q=2048, S_kv=32768, H=64, seed=1012, fp4=True),
    "mx4_2k_32k_h64_d128_zeros": dict(S_q=2048, S_kv=32768, H=64, zeros=True, fp4=True),
    "mx4_8k_64k_h64_d128_zeros": dict(S_q=8192, S_kv=65536, H=64, zeros=True, fp4=True),
}


def mx_config(name: str) -> MxDenseCase:
    kw = dict(MX_CONFIGS[name])
    fp4 = kw.pop("fp4", False)
    if kw.pop("zeros", False):
        return mx_zero_case(kw["S_q"], kw["S_kv"], kw["H"], fp4=fp4, name=name)
    return mx_dense_case(kw["S_q"], kw["S_kv"], kw["H"], seed=kw["seed"], fp4=fp4, name=name)


@dataclass
class PagedMxCase:
    """Paged decode input with MX (block-scaled) elements: E4M3 or packed E2M1
    keys in pages, one int32 of four UE8M0 scales per key slot and per
    (query row, head)."""
    name: str
    q: torch.Tensor            # [B*next_n, H, 128] uint8 (E4M3) or [.., 64] (E2M1 pairs)
    q_sf: torch.Tensor         # [B*next_n, H] int32
    kv_cache: torch.Tensor     # [num_blocks, block_kv, 128] or [.., 64] uint8
    kv_sf: torch.Tensor        # [num_blocks, block_kv] int32
    weights: torch.Tensor      # [B*next_n, H] float32
    context_lens: torch.Tensor  # [B] int32
    block_table: torch.Tensor  # [B, max_blocks_per_seq] int32
    next_n: int
    ldo: int
    fp4: bool
    D = 128
    clean = True

    @property
    def B(self):
        return self.context_lens.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def block_kv(self):
        return self.kv_cache.shape[1]

    @property
    def num_blocks(self):
        return self.kv_cache.shape[0]

    @property
    def max_blocks_per_seq(self):
        return self.block_table.shape[1]

    def valid_counts(self) -> torch.Tensor:
        ctx = self.context_lens.to(torch.int64).repeat_interleave(self.next_n)
        t = torch.arange(self.next_n, dtype=torch.int64).repeat(self.B)
        return (ctx - self.next_n + t + 1).clamp(min=0)


def paged_mx_case(B: int, next_n: int, H: int, *, seed: int, context_lens, block_kv: int = 64,
                  num_blocks: Optional[int] = None, fp4: bool = False, sf_lo: int = 124,
                  sf_hi: int = 130, max_blocks_per_seq: Optional[int] = None,
                  name: str = "paged_mx") -> PagedMxCase:
    """Paged MX case: the given context lengths, pages handed out by a random
    permutation of the blocks, elements as ``mx_dense_case``."""
    g = _gen(seed)
    ctx = torch.as_tensor(context_lens, dtype=torch.int64)
    pages = (ctx.clamp(min=0) + block_kv - 1) // block_kv
    max_blocks = max_blocks_per_seq or max(1, int(pages.max()))
    if num_blocks is None:
        num_blocks = int(pages.sum()) + 3
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(pages[b])
        table[b, :n] = perm[off:off + n]
        off += n
    D = 128
    if fp4:
        q, kv = e2m1_pairs((B * next_n, H, D // 2), g), e2m1_pairs((num_blocks, block_kv, D // 2), g)
    else:
        q, kv = e4m3_normal((B * next_n, H, D), g), e4m3_normal((num_blocks, block_kv, D), g)
    q_sf = packed_scales((B * next_n, H), sf_lo, sf_hi, g)
    kv_sf = packed_scales((num_blocks, block_kv), sf_lo, sf_hi, g)
    weights = torch.randn((B * next_n, H), generator=g)
    return PagedMxCase(name, q, q_sf, kv, kv_sf, weights, ctx.to(torch.int32), table, next_n,
                       max_blocks * block_kv, fp4)


# The paged decode shape with MX keys (MXFP8, and MXFP4: the FP4 keys of the
# "[PR #314] ..." page's paged test matrix): 64 sequences, next_n = 2, H = 64,
# contexts uniform in [4096, 65536], 64-key pages over a 70000-block pool.
PAGED_MX_CONFIGS = {
    "paged_mx_b64_n2_h64_d128": dict(fp4=False, seed=1013),
    "paged_mx4_b64_n2_h64_d128": dict(fp4=True, seed=1014),
}


def paged_mx_config(name: str) -> PagedMxCase:
    kw = PAGED_MX_CONFIGS[name]
    g = _gen(kw["seed"])
    ctx = torch.randint(4096, 65536 + 1, (64,), generator=g, dtype=torch.int64)
    return paged_mx_case(64, 2, 64, seed=kw["seed"] + 100, context_lens=ctx.tolist(), block_kv=64,
                         num_blocks=70000, fp4=kw["fp4"], max_blocks_per_seq=65536 // 64, name=name)
