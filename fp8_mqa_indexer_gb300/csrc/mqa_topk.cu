// mqa_topk.cu -- top-k key selection over rows of MQA logits.
//
// For each query row: the topk keys of the row's range with the largest
// logits, in ascending key order, padded with -1.  This is the `indices`
// input of the sparse-attention call on the "FlashMLA" page (parameters of
// flash_mla_with_kvcache: shape (batch, seq_len_q, topk), invalid entries
// -1).  Larger means later in the IEEE-754 totalOrder of the fp32 value;
// among equal values the smaller key is taken, so the result is unique.
//
// A persistent grid (four CTAs per SM) walks the rows, one row per CTA at a
// time.  A block-wide step covers four tiles of 4 x 256 elements; a thread
// loads four consecutive elements of each tile (coalesced 16-byte loads, four
// in flight per thread).  Each logit maps to a 32-bit key whose unsigned
// order is totalOrder, and a radix select over three digits (bits 31..20,
// 19..8, 7..0) finds the k-th largest key T:
//   0. (rows with k <= 2048 and at least max(8192, 4 k) keys) a sample of
//      1/16 of the row (whole 128-byte lines, one in every 16) sets a
//      threshold t0 that about 1.4 k keys clear; one ordered pass compacts
//      every key >= t0 into shared memory and, when that list holds between k
//      and its capacity of keys, the selection runs on the list alone, with
//      two 12-bit digits of key - t0 in place of steps 1 to 3 (the list's keys
//      spread over those digits, so their histogram atomics rarely collide,
//      where the absolute digit 1 of keys near t0 falls in a few bins): the
//      row is read from HBM once.  Otherwise:
//   1. histogram of digit 1 over the row (the row's read from HBM) gives the
//      bin holding the k-th largest key;
//   2. every element in or above that bin is compacted, in key order, into
//      shared memory (a second read of the row, from L2: the first read marks
//      the row's lines evict-last, the second evict-first);
//   3. histograms of digits 2 and 3 over the compacted elements of the bin
//      give T, the count of keys above T, and r = the number of keys equal to
//      T that are taken (the r smallest such keys);
//   4. one ordered pass over the compacted list writes each taken key at its
//      rank: (keys above T before it) + min(keys equal to T before it, r).
// If the bin and everything above it do not fit shared memory (many equal or
// nearly equal logits), steps 3 and 4 read the row from global memory.
// Rows with at most topk keys take every key without reading the logits.
#include <atomic>

#include "topk.h"

namespace mqa {
namespace {

constexpr int kNT = kTopkThreads;
constexpr int kNW = kNT / 32;
constexpr int kPer = 16;            // elements per thread per step: 4 tiles x 4
constexpr int kTile = 4 * kNT;      // elements per tile
constexpr int kStep = kPer * kNT;   // elements per block-wide step (4 tiles)
constexpr int kBins12 = 4096;       // digits 1 and 2
constexpr int kBins8 = 256;         // digit 3
constexpr int kCap = 4096;          // compacted elements held in shared memory
static_assert(kTile < (1 << 16), "per-tile counts are packed in 16-bit fields");

struct TopkSmem {
    alignas(16) unsigned hist[kBins12];
    alignas(16) unsigned cand_key[kCap];
    alignas(16) int cand_idx[kCap];
    unsigned warp_sum[2][kNW];
    unsigned long long warp_sum64[2][2][kNW];
    unsigned sel_bin, sel_above, sel_count;
};

// Unsigned key whose order is the IEEE-754 totalOrder of v: negative values
// have every bit flipped, non-negative ones only the sign bit.
__device__ __forceinline__ unsigned order_key(float v)
{
    const unsigned u = __float_as_uint(v);
    return u ^ ((unsigned)((int)u >> 31) | 0x80000000u);
}

// L2 eviction policies for the two reads of a row.
__device__ __forceinline__ unsigned long long policy_evict_last()
{
    unsigned long long p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ unsigned long long policy_evict_first()
{
    unsigned long long p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ float4 load4(const float* ptr, unsigned long long pol)
{
    float4 v;
    asm("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(ptr), "l"(pol));
    return v;
}

__device__ __forceinline__ float4 load4(const float* ptr)
{
    return __ldg(reinterpret_cast<const float4*>(ptr));
}

// Exclusive prefix sum of v over the block in thread order; `total` gets the
// block-wide sum.  One __syncthreads; callers alternate between the two
// warp_sum buffers, so a call's writes never meet the previous call's reads.
__device__ __forceinline__ unsigned block_exclusive_sum(unsigned v, unsigned* ws, unsigned& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        ws[warp] = x;
    __syncthreads();
    unsigned before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
        const unsigned s = ws[w];
        before += w < warp ? s : 0u;
        all += s;
    }
    total = all;
    return before + x - v;
}

// Exclusive prefix sums, in thread order, of two packed vectors of four 16-bit
// counts (one field per tile of a step); tot_* get the block-wide sums.  One
// __syncthreads, double-buffered like block_exclusive_sum.
__device__ __forceinline__ void block_exclusive_sum64x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long (*ws)[kNW],
                                                        unsigned long long& pre_a,
                                                        unsigned long long& pre_b,
                                                        unsigned long long& tot_a,
                                                        unsigned long long& tot_b)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = a, y = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long xs = __shfl_up_sync(0xffffffffu, x, o);
        const unsigned long long ys = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) {
            x += xs;
            y += ys;
        }
    }
    if (lane == 31) {
        ws[0][warp] = x;
        ws[1][warp] = y;
    }
    __syncthreads();
    unsigned long long ba = 0, bb = 0, ta = 0, tb = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
        const unsigned long long sa = ws[0][w], sb = ws[1][w];
        ba += w < warp ? sa : 0ull;
        bb += w < warp ? sb : 0ull;
        ta += sa;
        tb += sb;
    }
    pre_a = ba + x - a;
    pre_b = bb + y - b;
    tot_a = ta;
    tot_b = tb;
}

// Start, in index order, of each tile's run of a thread: the elements of all
// earlier tiles of the step plus those of earlier threads in this tile.
__device__ __forceinline__ void tile_offsets(unsigned long long pre, unsigned long long tot,
                                             unsigned (&off)[4])
{
    unsigned before = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        off[g] = before + (unsigned)((pre >> (16 * g)) & 0xffffu);
        before += (unsigned)((tot >> (16 * g)) & 0xffffu);
    }
}

// The bin of hist[0, NBINS) that holds the need-th largest element (1 <= need
// <= the histogram's total): its index, the elements in higher bins and the
// elements in the bin.  Ends with the selection visible to all threads.  The
// histogram is sm.hist unless `hist` names another shared array.
template <int NBINS>
__device__ __forceinline__ void select_bin(TopkSmem& sm, unsigned need, int& buf, unsigned& bin,
                                           unsigned& above, unsigned& count,
                                           const unsigned* hist = nullptr)
{
    const unsigned* hs = hist ? hist : sm.hist;
    constexpr int kB = NBINS >= kNT ? NBINS / kNT : 1;   // bins per thread
    static_assert(kB == 1 || kB % 4 == 0, "bins are read four at a time");
    const int b0 = threadIdx.x * kB;
    unsigned h[kB], s = 0;
    if constexpr (kB == 1) {
        h[0] = b0 < NBINS ? hs[b0] : 0u;
    } else {
#pragma unroll
        for (int q = 0; q < kB; q += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(&hs[b0 + q]);
            h[q] = v.x, h[q + 1] = v.y, h[q + 2] = v.z, h[q + 3] = v.w;
        }
    }
#pragma unroll
    for (int q = 0; q < kB; ++q)
        s += h[q];
    unsigned total;
    const unsigned before = block_exclusive_sum(s, sm.warp_sum[buf], total);
    buf ^= 1;
    unsigned acc = total - before - s;   // elements in the bins of higher threads
    if (acc < need && acc + s >= need) {  // the one thread whose bins hold it
#pragma unroll
        for (int q = kB - 1; q >= 0; --q) {
            if (acc < need && acc + h[q] >= need) {
                sm.sel_bin = (unsigned)(b0 + q);
                sm.sel_above = acc;
                sm.sel_count = h[q];
            }
            acc += h[q];
        }
    }
    __syncthreads();
    bin = sm.sel_bin;
    above = sm.sel_above;
    count = sm.sel_count;
}

// The row's range as columns of its logits row.
struct RowView {
    const float* ptr;      // column 0
    long long c_lo, c_hi;  // columns of the range
    long long c_start;     // c_lo rounded down to a 16-byte aligned address
    int key_of_col0;       // key index = column + key_of_col0
};

// Element e = 4 g + j of a thread's step is element j of its run in tile g.
struct RowIdx {            // key of element e in the row
    int key0;              // key of the thread's first element in tile 0
    __device__ int operator()(int e) const { return key0 + (e >> 2) * kTile + (e & 3); }
};

struct CandIdx {           // key of element e in the compacted list
    const int* p;          // the thread's first entry in tile 0
    __device__ int operator()(int e) const { return p[(e >> 2) * kTile + (e & 3)]; }
};

// f(key[16], okmask, idx) for every block-wide step over the range: element
// 4 g + j of thread t is column base + g * kTile + 4 t + j.  All threads take
// the same number of steps, so f may synchronize the block.  Whole aligned
// runs load as float4 with L2 policy `pol`, the ragged ends element by element.
template <bool HINT, class F>
__device__ __forceinline__ void for_row(const RowView& r, unsigned long long pol, F&& f)
{
    for (long long base = r.c_start; base < r.c_hi; base += kStep) {
        const long long c0 = base + 4 * threadIdx.x;
        float v[kPer];
        if (base >= r.c_lo && base + kStep <= r.c_hi) {   // the whole step is in range
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 x = HINT ? load4(r.ptr + c0 + g * kTile, pol) : load4(r.ptr + c0 + g * kTile);
                v[4 * g] = x.x, v[4 * g + 1] = x.y, v[4 * g + 2] = x.z, v[4 * g + 3] = x.w;
            }
            unsigned key[kPer];
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                key[e] = order_key(v[e]);
            f(key, (1u << kPer) - 1u, RowIdx{(int)c0 + r.key_of_col0});
            continue;
        }
        unsigned okm = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const long long c = c0 + g * kTile;
            if (c >= r.c_lo && c + 4 <= r.c_hi) {
                const float4 x = HINT ? load4(r.ptr + c, pol) : load4(r.ptr + c);
                v[4 * g] = x.x, v[4 * g + 1] = x.y, v[4 * g + 2] = x.z, v[4 * g + 3] = x.w;
                okm |= 0xfu << (4 * g);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool ok = c + j >= r.c_lo && c + j < r.c_hi;
                    v[4 * g + j] = ok ? __ldg(r.ptr + c + j) : 0.f;
                    okm |= (unsigned)ok << (4 * g + j);
                }
            }
        }
        unsigned key[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            key[e] = order_key(v[e]);
        f(key, okm, RowIdx{(int)c0 + r.key_of_col0});
    }
}

// The same over the first m compacted elements, in key order (entry
// base + g * kTile + 4 t + j).
template <class F>
__device__ __forceinline__ void for_cand(const TopkSmem& sm, unsigned m, F&& f)
{
    for (unsigned base = 0; base < m; base += kStep) {
        const unsigned k0 = base + 4 * threadIdx.x;
        unsigned key[kPer], okm = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const unsigned k = k0 + g * kTile;
            const uint4 v = k < (unsigned)kCap ? *reinterpret_cast<const uint4*>(&sm.cand_key[k])
                                               : make_uint4(0u, 0u, 0u, 0u);
            key[4 * g] = v.x, key[4 * g + 1] = v.y, key[4 * g + 2] = v.z, key[4 * g + 3] = v.w;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                okm |= (unsigned)(k + j < m) << (4 * g + j);
        }
        f(key, okm, CandIdx{sm.cand_idx + (k0 < (unsigned)kCap ? k0 : 0u)});
    }
}

template <int NBINS>
__device__ __forceinline__ void clear_hist(TopkSmem& sm)
{
    uint4* h4 = reinterpret_cast<uint4*>(sm.hist);
    for (int b = threadIdx.x; b < NBINS / 4; b += kNT)
        h4[b] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
}

template <class Walk>
__device__ __forceinline__ void write_selected(TopkSmem& sm, Walk&& each, unsigned T, unsigned r,
                                               unsigned k, int* out, int& buf);

// Digits 2 and 3 over `each` (a row or list walk), then the ordered write of
// the selection.  b1 / above1 come from digit 1.
template <class Walk>
__device__ __forceinline__ void finish_row(TopkSmem& sm, Walk&& each, unsigned b1, unsigned above1,
                                           unsigned k, int* out, int& buf)
{
    clear_hist<kBins12>(sm);
    each([&](const unsigned(&key)[kPer], unsigned okm, auto) {
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if (((okm >> e) & 1u) && (key[e] >> 20) == b1)
                atomicAdd(&sm.hist[(key[e] >> 8) & 0xfffu], 1u);
    });
    __syncthreads();
    unsigned b2, above2, cnt;
    select_bin<kBins12>(sm, k - above1, buf, b2, above2, cnt);
    const unsigned prefix = (b1 << 12) | b2;
    clear_hist<kBins8>(sm);
    each([&](const unsigned(&key)[kPer], unsigned okm, auto) {
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if (((okm >> e) & 1u) && (key[e] >> 8) == prefix)
                atomicAdd(&sm.hist[key[e] & 0xffu], 1u);
    });
    __syncthreads();
    unsigned b3, above3;
    select_bin<kBins8>(sm, k - above1 - above2, buf, b3, above3, cnt);
    const unsigned T = (prefix << 8) | b3;
    write_selected(sm, each, T, k - above1 - above2 - above3, k, out, buf);
}

// The ordered write of a selection: every key above T, and the first r keys
// equal to T, each at its rank in key order: (keys above T before it) +
// min(keys equal to T before it, r).
template <class Walk>
__device__ __forceinline__ void write_selected(TopkSmem& sm, Walk&& each, unsigned T, unsigned r,
                                               unsigned k, int* out, int& buf)
{
    unsigned gt_run = 0, eq_run = 0;
    each([&](const unsigned(&key)[kPer], unsigned okm, auto idx) {
        unsigned gm = 0, qm = 0;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const bool ok = (okm >> e) & 1u;
            gm |= (unsigned)(ok && key[e] > T) << e;
            qm |= (unsigned)(ok && key[e] == T) << e;
        }
        unsigned long long ga = 0, qa = 0;   // per-tile counts, 16 bits each
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            ga |= (unsigned long long)__popc((gm >> (4 * g)) & 0xfu) << (16 * g);
            qa |= (unsigned long long)__popc((qm >> (4 * g)) & 0xfu) << (16 * g);
        }
        unsigned long long gpre, qpre, gtot, qtot;
        block_exclusive_sum64x2(ga, qa, sm.warp_sum64[buf], gpre, qpre, gtot, qtot);
        buf ^= 1;
        unsigned goff[4], qoff[4];
        tile_offsets(gpre, gtot, goff);
        tile_offsets(qpre, qtot, qoff);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            unsigned gb = gt_run + goff[g], eb = eq_run + qoff[g];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = 4 * g + j;
                if ((gm >> e) & 1u) {
                    const unsigned pos = gb + min(eb, r);
                    if (pos < k)
                        out[pos] = idx(e);
                    ++gb;
                } else if ((qm >> e) & 1u) {
                    if (eb < r && gb + eb < k)
                        out[gb + eb] = idx(e);
                    ++eb;
                }
            }
        }
        unsigned gsum = 0, qsum = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            gsum += (unsigned)((gtot >> (16 * g)) & 0xffffu);
            qsum += (unsigned)((qtot >> (16 * g)) & 0xffffu);
        }
        gt_run += gsum;
        eq_run += qsum;
    });
}

// Ordered compaction of the walk's elements with key >= thr into the shared
// list (the first kCap of them, in key order); returns how many there are.
template <class Walk>
__device__ __forceinline__ unsigned compact_walk(TopkSmem& sm, Walk&& each, unsigned thr, int& buf)
{
    unsigned run = 0;
    each([&](const unsigned(&key)[kPer], unsigned okm, auto idx) {
        unsigned fm = 0;
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            fm |= (unsigned)(((okm >> e) & 1u) && key[e] >= thr) << e;
        unsigned long long fa = 0;   // per-tile counts, 16 bits each
#pragma unroll
        for (int g = 0; g < 4; ++g)
            fa |= (unsigned long long)__popc((fm >> (4 * g)) & 0xfu) << (16 * g);
        unsigned long long pre, unused_pre, tot, unused_tot;
        block_exclusive_sum64x2(fa, 0ull, sm.warp_sum64[buf], pre, unused_pre, tot, unused_tot);
        buf ^= 1;
        unsigned off[4];
        tile_offsets(pre, tot, off);
        if (fm) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                unsigned pos = run + off[g];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int e = 4 * g + j;
                    if ((fm >> e) & 1u) {
                        if (pos < (unsigned)kCap) {
                            sm.cand_key[pos] = key[e];
                            sm.cand_idx[pos] = idx(e);
                        }
                        ++pos;
                    }
                }
            }
        }
        unsigned sum = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g)
            sum += (unsigned)((tot >> (16 * g)) & 0xffffu);
        run += sum;
    });
    __syncthreads();
    return run;
}

template <bool HINT>
__device__ __forceinline__ unsigned compact_row(TopkSmem& sm, const RowView& r,
                                                unsigned long long pol, unsigned thr, int& buf)
{
    return compact_walk(
        sm, [&](auto&& f) { for_row<HINT>(r, pol, f); }, thr, buf);
}

// Element e (0..15) of v, by a four-level select on the bits of e (no local
// memory for a dynamic register index).
__device__ __forceinline__ float pick16(const float (&v)[16], unsigned e)
{
    float a[8], b[4], c[2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = (e & 1u) ? v[2 * i + 1] : v[2 * i];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        b[i] = (e & 2u) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
    for (int i = 0; i < 2; ++i)
        c[i] = (e & 4u) ? b[2 * i + 1] : b[2 * i];
    return (e & 8u) ? c[1] : c[0];
}

// Ordered compaction of the row's keys >= thr into the shared list (the one-
// pass case): each thread owns 16 consecutive columns of a block-wide step
// (four 16-byte loads), so the order of the list is the thread order and one
// 32-bit block scan per step places every thread's keys.  For thr at or above
// the key of +0, key(v) >= thr is a signed compare of v's raw bits with thr's
// magnitude bits (negative values fail; non-negative ones order as their
// bits); keys are formed only for the elements taken.  Returns the number of
// keys found (entries past kCap are counted, not written).
__device__ __forceinline__ unsigned compact_row_owned(TopkSmem& sm, const RowView& r, unsigned thr,
                                                      int& buf)
{
    const bool fast = thr >= 0x80000000u;
    const int ithr = (int)(thr & 0x7fffffffu);
    unsigned run = 0;
    for (long long base = r.c_start; base < r.c_hi; base += kStep) {
        const long long c0 = base + 16 * (long long)threadIdx.x;
        float v[16];
        unsigned fm = 0;
        if (c0 >= r.c_lo && c0 + 16 <= r.c_hi) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 x = load4(r.ptr + c0 + 4 * q);
                v[4 * q] = x.x, v[4 * q + 1] = x.y, v[4 * q + 2] = x.z, v[4 * q + 3] = x.w;
            }
            if (fast) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    fm |= (unsigned)((int)__float_as_uint(v[e]) >= ithr) << e;
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    fm |= (unsigned)(order_key(v[e]) >= thr) << e;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const bool ok = c0 + e >= r.c_lo && c0 + e < r.c_hi;
                v[e] = ok ? __ldg(r.ptr + c0 + e) : 0.f;
                fm |= (unsigned)(ok && order_key(v[e]) >= thr) << e;
            }
        }
        unsigned total;
        unsigned pos = run + block_exclusive_sum(__popc(fm), sm.warp_sum[buf], total);
        buf ^= 1;
        const int idx0 = (int)c0 + r.key_of_col0;
        while (fm) {
            const unsigned e = __ffs(fm) - 1;
            fm &= fm - 1;
            if (pos < (unsigned)kCap) {
                sm.cand_key[pos] = order_key(pick16(v, e));
                sm.cand_idx[pos] = idx0 + (int)e;
            }
            ++pos;
        }
        run += total;
    }
    __syncthreads();
    return run;
}

// Threshold key t0 from a sample of the row (one aligned float4 in every
// `stride` elements, 1/16 of the keys for rows up to 65536): the lower edge of
// the 24-bit key prefix holding the sample's need-th largest key, with need
// scaled so that about 1.4 k keys of the whole row lie at or above t0.  The
// sample only steers the work: whatever t0 is, the caller checks the count
// it yields and falls back to the full selection.  Returns false when the
// sample is too small.  Uses the shared list as scratch.
__device__ __forceinline__ bool sample_threshold(TopkSmem& sm, const RowView& r, unsigned n,
                                                 unsigned k, int& buf, unsigned& t0)
{
    // whole 128-byte lines (8 float4), one line in every 8 * stride elements
    const long long c128 =
        r.c_lo - (long long)((reinterpret_cast<unsigned long long>(r.ptr + r.c_lo) >> 2) & 31);
    const long long span = r.c_hi - c128;
    long long stride = 64;
    while (((span + 8 * stride - 1) / (8 * stride)) * 8 > kCap / 4)
        stride *= 2;
    const int nf4 = (int)(((span + 8 * stride - 1) / (8 * stride)) * 8);
    clear_hist<kBins12>(sm);
    unsigned valid = 0;
    for (int f = threadIdx.x; f < nf4; f += kNT) {
        const long long c = c128 + (long long)(f >> 3) * (8 * stride) + 4 * (f & 7);
        uint4 kk = make_uint4(0u, 0u, 0u, 0u);   // key 0: not a sample
        if (c >= r.c_lo && c + 4 <= r.c_hi) {
            const float4 x = load4(r.ptr + c);
            kk = make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
            atomicAdd(&sm.hist[kk.x >> 20], 1u);
            atomicAdd(&sm.hist[kk.y >> 20], 1u);
            atomicAdd(&sm.hist[kk.z >> 20], 1u);
            atomicAdd(&sm.hist[kk.w >> 20], 1u);
            valid += 4;
        }
        *reinterpret_cast<uint4*>(&sm.cand_key[4 * f]) = kk;
    }
    unsigned total;
    block_exclusive_sum(valid, sm.warp_sum[buf], total);   // also orders the atomics
    buf ^= 1;
    if (total < 256)
        return false;
    unsigned long long want = (14ull * k * total + 10ull * n - 1) / (10ull * n);
    const unsigned need = want < 1 ? 1u : (want > total ? total : (unsigned)want);
    unsigned b1, above1, cnt1;
    select_bin<kBins12>(sm, need, buf, b1, above1, cnt1);
    clear_hist<kBins12>(sm);
    for (int f = threadIdx.x; f < nf4; f += kNT) {
        const uint4 kk = *reinterpret_cast<const uint4*>(&sm.cand_key[4 * f]);
        const unsigned kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (kv[j] != 0u && (kv[j] >> 20) == b1)
                atomicAdd(&sm.hist[(kv[j] >> 8) & 0xfffu], 1u);
    }
    __syncthreads();
    unsigned b2, above2, cnt2;
    select_bin<kBins12>(sm, need - above1, buf, b2, above2, cnt2);
    t0 = (b1 << 20) | (b2 << 8);
    return true;
}

// Exact selection from the first m list entries (in key order), all of them
// keys >= t0, when the k-th largest lies below t0 + 2^24 - 4096: two 12-bit
// digits of key - t0 (the first clamped to 4095) instead of three absolute
// ones.  The list's keys are spread over the relative digits, so the
// histogram atomics rarely collide.  Returns false, having written nothing,
// when the k-th largest falls in the clamped bin.
__device__ __forceinline__ bool select_from_list_rel(TopkSmem& sm, unsigned m, unsigned k,
                                                     unsigned t0, int* out, int& buf)
{
    auto d1 = [t0](unsigned key) { return min((key - t0) >> 12, (unsigned)(kBins12 - 1)); };
    clear_hist<kBins12>(sm);
    for_cand(sm, m, [&](const unsigned(&key)[kPer], unsigned okm, auto) {
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if ((okm >> e) & 1u)
                atomicAdd(&sm.hist[d1(key[e])], 1u);
    });
    __syncthreads();
    unsigned c1, above1, n1;
    select_bin<kBins12>(sm, k, buf, c1, above1, n1);
    if (c1 == kBins12 - 1)
        return false;
    clear_hist<kBins12>(sm);
    for_cand(sm, m, [&](const unsigned(&key)[kPer], unsigned okm, auto) {
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if (((okm >> e) & 1u) && d1(key[e]) == c1)
                atomicAdd(&sm.hist[(key[e] - t0) & 0xfffu], 1u);
    });
    __syncthreads();
    unsigned c2, above2, n2;
    select_bin<kBins12>(sm, k - above1, buf, c2, above2, n2);
    write_selected(
        sm, [&](auto&& f) { for_cand(sm, m, f); }, t0 + (c1 << 12) + c2, k - above1 - above2, k, out,
        buf);
    return true;
}

// Exact selection from the first m list entries (in key order), which hold
// every key of the row that can be among its k largest (k <= m <= kCap).
__device__ __forceinline__ void select_from_list(TopkSmem& sm, unsigned m, unsigned k, int* out,
                                                 int& buf)
{
    clear_hist<kBins12>(sm);
    for_cand(sm, m, [&](const unsigned(&key)[kPer], unsigned okm, auto) {
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if ((okm >> e) & 1u)
                atomicAdd(&sm.hist[key[e] >> 20], 1u);
    });
    __syncthreads();
    unsigned b1, above1, n1;
    select_bin<kBins12>(sm, k, buf, b1, above1, n1);
    finish_row(
        sm, [&](auto&& f) { for_cand(sm, m, f); }, b1, above1, k, out, buf);
}

__global__ void __launch_bounds__(kNT, kTopkCtasPerSm) topk_kernel(TopkParams p)
{
    extern __shared__ __align__(16) unsigned char topk_smem_raw[];
    TopkSmem& sm = *reinterpret_cast<TopkSmem*>(topk_smem_raw);
    int buf = 0;
    const unsigned k = (unsigned)p.topk;
    const unsigned long long keep = policy_evict_last(), drop = policy_evict_first();
    for (int i = blockIdx.x; i < p.rows; i += gridDim.x) {
        // ---- the row's key range, intersected with [0, n_cols)
        long long lo, hi;
        if (p.context_lens) {
            const int b = i / p.next_n, t = i % p.next_n;
            lo = 0;
            hi = (long long)__ldg(p.context_lens + b) - p.next_n + t + 1;
        } else {
            lo = __ldg(p.k_start + i);
            hi = __ldg(p.k_end + i);
        }
        lo = lo < 0 ? 0 : (lo > p.n_cols ? p.n_cols : lo);
        hi = hi > p.n_cols ? p.n_cols : hi;
        hi = hi < lo ? lo : hi;
        if (p.compressed && hi - lo > p.ldo)
            hi = lo + p.ldo;
        const unsigned n = (unsigned)(hi - lo);
        int* out = p.indices + (long long)i * p.topk;
        const unsigned taken = n < k ? n : k;
        __syncthreads();   // the previous row's shared state is no longer read
        if (n <= k) {
            for (unsigned c = threadIdx.x; c < n; c += kNT)
                out[c] = (int)(lo + c);
        } else {
            RowView r;
            r.ptr = p.logits + (long long)i * p.ldo;
            r.c_lo = p.compressed ? 0 : lo;
            r.c_hi = r.c_lo + (long long)n;
            r.key_of_col0 = p.compressed ? (int)lo : 0;
            r.c_start = r.c_lo - (long long)((reinterpret_cast<unsigned long long>(r.ptr + r.c_lo) >> 2) & 3);
            bool done = false;
            // ---- common case: a sampled threshold, one pass over the row
            unsigned t0;
            if (2u * k <= (unsigned)kCap && n >= 8192u && n >= 4u * k &&
                sample_threshold(sm, r, n, k, buf, t0)) {
                const unsigned m = compact_row_owned(sm, r, t0, buf);
                if (m >= k && m <= (unsigned)kCap) {
                    if (!select_from_list_rel(sm, m, k, t0, out, buf))
                        select_from_list(sm, m, k, out, buf);
                    done = true;
                }
            }
            if (!done) {
                // ---- full selection: digit 1 over the row
                clear_hist<kBins12>(sm);
                for_row<true>(r, keep, [&](const unsigned(&key)[kPer], unsigned okm, RowIdx) {
#pragma unroll
                    for (int e = 0; e < kPer; ++e)
                        if ((okm >> e) & 1u)
                            atomicAdd(&sm.hist[key[e] >> 20], 1u);
                });
                __syncthreads();
                unsigned b1, above1, n1;
                select_bin<kBins12>(sm, k, buf, b1, above1, n1);
                const unsigned m = above1 + n1;   // elements in bin b1 or above
                if (m <= (unsigned)kCap) {
                    // ---- compact those elements, in key order, into shared memory
                    const unsigned mm = compact_row<true>(sm, r, drop, b1 << 20, buf);
                    finish_row(
                        sm, [&](auto&& f) { for_cand(sm, mm < (unsigned)kCap ? mm : (unsigned)kCap, f); },
                        b1, above1, k, out, buf);
                } else {
                    finish_row(
                        sm, [&](auto&& f) { for_row<true>(r, drop, f); }, b1, above1, k, out, buf);
                }
            }
        }
        for (unsigned c = taken + threadIdx.x; c < k; c += kNT)
            out[c] = -1;
    }
}

// ------------------------------------------------ fused logits + top-k
// The candidate form of a row with range [lo, hi) split at s: keys [s, hi)
// (the prefix) have their logits at their own columns; line L of [lo, s) (the
// remainder; keys [32 L, 32 L + 32)) holds, packed at its front in key order,
// the logits of the keys whose bits are set in the line's mask.
struct CandView {
    const float* vals;      // the row's values
    const unsigned* mask;   // the row's line masks
    long long c_lo, c_hi;   // the row's key range
    long long s;            // first prefix key (a multiple of 128, or c_lo)
    unsigned thr;           // prefix keys below thr are not taken
};

// f(key[16], okmask, idx) over the candidate row, element 4 g + j of thread t
// being key base + g * kTile + 4 t + j as in for_row (a run of four keys never
// crosses a line; it crosses s only when s = c_lo, the row having no
// remainder).  Remainder keys without a candidate and prefix keys below thr
// are not ok; remainder mask bits are only ever set for keys of the row's
// range.
template <class F>
__device__ __forceinline__ void for_cand_row(const CandView& r, F&& f)
{
    for (long long base = r.c_lo & ~31ll; base < r.c_hi; base += kStep) {
        const long long c0 = base + 4 * threadIdx.x;
        unsigned m[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {   // the step's remainder masks first
            const long long c = c0 + g * kTile;
            m[g] = (c + 4 > r.c_lo && c + 4 <= r.s) ? __ldg(r.mask + (c >> 5)) : 0u;
        }
        unsigned key[kPer], okm = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const long long c = c0 + g * kTile;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                key[4 * g + j] = 0u;
            if (c + 4 > r.s) {   // prefix: plain logits
                if (c >= r.s && c + 4 <= r.c_hi) {
                    const float4 x = load4(r.vals + c);
                    key[4 * g] = order_key(x.x), key[4 * g + 1] = order_key(x.y);
                    key[4 * g + 2] = order_key(x.z), key[4 * g + 3] = order_key(x.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        okm |= (unsigned)(key[4 * g + j] >= r.thr) << (4 * g + j);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (c + j >= r.s && c + j < r.c_hi) {
                            key[4 * g + j] = order_key(__ldg(r.vals + c + j));
                            okm |= (unsigned)(key[4 * g + j] >= r.thr) << (4 * g + j);
                        }
                    }
                }
            } else {   // remainder: candidates packed at the front of the line
                const int pos = (int)(c & 31);
                const float* line = r.vals + (c & ~31ll);
                const unsigned bits = (m[g] >> pos) & 0xfu;
                unsigned rank = __popc(m[g] & ((1u << pos) - 1u));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if ((bits >> j) & 1u) {
                        key[4 * g + j] = order_key(__ldg(line + rank));
                        ++rank;
                        okm |= 1u << (4 * g + j);
                    }
                }
            }
        }
        f(key, okm, RowIdx{(int)c0});
    }
}

// Row i's key range, clamped to [0, n_cols] as the top-k kernel clamps it.
__device__ __forceinline__ void cand_range(const CandTopkParams& p, int i, int& lo, int& hi)
{
    long long a = __ldg(p.k_start + i), b = __ldg(p.k_end + i);
    a = a < 0 ? 0 : (a > p.n_cols ? p.n_cols : a);
    b = b > p.n_cols ? p.n_cols : b;
    b = b < a ? a : b;
    lo = (int)a;
    hi = (int)b;
}

// Prefix and remainder of each row.  The prefix holds at least
// max(2 topk, sqrt(n topk)) keys: about the length that minimises the
// candidates written (all of the prefix, plus about topk / prefix of the
// remainder for logits in random order).
__global__ void cand_split_kernel(CandTopkParams p)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.rows)
        return;
    int lo, hi;
    cand_range(p, i, lo, hi);
    const long long n = (long long)hi - lo, k = p.topk;
    int pre_lo = lo, pre_hi = lo, rem_hi = lo;
    if (n > k) {
        long long len = (long long)ceil(sqrt((double)n * (double)k));
        len = len < 2 * k ? 2 * k : len;
        len = (len + 127) & ~127ll;
        const long long s = ((long long)hi - len) & ~127ll;   // rounds toward -inf
        pre_lo = s > lo ? (int)s : lo;
        pre_hi = hi;
        rem_hi = pre_lo;
    }
    p.pre_lo[i] = pre_lo;
    p.pre_hi[i] = pre_hi;
    p.rem_lo[i] = lo;
    p.rem_hi[i] = rem_hi;
    p.thr[i] = 0u;
    p.thr_f[i] = __int_as_float(0xff800000);   // -inf
    p.t0[i] = 0u;
}

// thr[i] = order key T of the topk-th largest logit of row i's prefix and
// thr_f[i] = that logit, for rows with a remainder (the prefix then holds more
// than topk keys, every one of them written at its own column): digits 1 to 3
// of the radix select, each over the prefix.  The same histograms give t0[i],
// the lower edge of the 24-bit key prefix holding the prefix's need-th largest
// logit, need scaled so that about 1.4 topk keys of the whole row lie at or
// above t0 when the prefix is typical of the row (0: no such estimate).  t0
// only steers the selection, which checks the count it yields.
__global__ void __launch_bounds__(kNT, kTopkCtasPerSm) cand_threshold_kernel(CandTopkParams p)
{
    extern __shared__ __align__(16) unsigned char topk_smem_raw[];
    TopkSmem& sm = *reinterpret_cast<TopkSmem*>(topk_smem_raw);
    unsigned* hist2 = sm.cand_key;   // a second 4096-bin histogram
    int buf = 0;
    const unsigned k = (unsigned)p.topk;
    for (int i = blockIdx.x; i < p.rows; i += gridDim.x) {
        const int lo = __ldg(p.rem_lo + i), s = __ldg(p.rem_hi + i);
        if (s <= lo)
            continue;   // the same for every thread of the block
        __syncthreads();   // the previous row's shared state is no longer read
        RowView r;
        r.ptr = p.vals + (long long)i * p.ldo;
        r.c_lo = s;
        r.c_hi = __ldg(p.pre_hi + i);
        r.key_of_col0 = 0;
        r.c_start = r.c_lo - (long long)((reinterpret_cast<unsigned long long>(r.ptr + r.c_lo) >> 2) & 3);
        const unsigned long long pre_n = (unsigned long long)(r.c_hi - r.c_lo);
        const unsigned long long row_n = (unsigned long long)(r.c_hi - lo);
        const unsigned long long want = (14ull * k * pre_n + 10ull * row_n - 1) / (10ull * row_n);
        const unsigned need = want < 1 ? 1u : (unsigned)want;
        const bool est = need < k;
        auto each = [&](auto&& f) { for_row<false>(r, 0ull, f); };
        clear_hist<kBins12>(sm);
        each([&](const unsigned(&key)[kPer], unsigned okm, RowIdx) {
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                if ((okm >> e) & 1u)
                    atomicAdd(&sm.hist[key[e] >> 20], 1u);
        });
        __syncthreads();
        unsigned b1, above1, n1, c1 = 0, cabove1 = 0, cn1 = 0;
        select_bin<kBins12>(sm, k, buf, b1, above1, n1);
        if (est)
            select_bin<kBins12>(sm, need, buf, c1, cabove1, cn1);
        clear_hist<kBins12>(sm);
        for (int b = threadIdx.x; b < kBins12 / 4; b += kNT)
            reinterpret_cast<uint4*>(hist2)[b] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        each([&](const unsigned(&key)[kPer], unsigned okm, RowIdx) {
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                if (((okm >> e) & 1u) && (key[e] >> 20) == b1)
                    atomicAdd(&sm.hist[(key[e] >> 8) & 0xfffu], 1u);
                if (est && ((okm >> e) & 1u) && (key[e] >> 20) == c1)
                    atomicAdd(&hist2[(key[e] >> 8) & 0xfffu], 1u);
            }
        });
        __syncthreads();
        unsigned b2, above2, n2, c2 = 0, cabove2 = 0, cn2 = 0;
        select_bin<kBins12>(sm, k - above1, buf, b2, above2, n2);
        if (est)
            select_bin<kBins12>(sm, need - cabove1, buf, c2, cabove2, cn2, hist2);
        const unsigned prefix = (b1 << 12) | b2;
        clear_hist<kBins8>(sm);
        each([&](const unsigned(&key)[kPer], unsigned okm, RowIdx) {
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                if (((okm >> e) & 1u) && (key[e] >> 8) == prefix)
                    atomicAdd(&sm.hist[key[e] & 0xffu], 1u);
        });
        __syncthreads();
        unsigned b3, above3, n3;
        select_bin<kBins8>(sm, k - above1 - above2, buf, b3, above3, n3);
        if (threadIdx.x == 0) {
            const unsigned T = (prefix << 8) | b3;
            p.thr[i] = T;
            // the logit whose order key is T (order_key inverted)
            p.thr_f[i] = __uint_as_float((T & 0x80000000u) ? (T ^ 0x80000000u) : ~T);
            p.t0[i] = est ? (c1 << 20) | (c2 << 8) : 0u;
        }
    }
}

// The topk largest candidates of each row, in ascending key order, -1 padded.
// The candidates hold every logit of the row with order key >= thr[i] (the
// prefix's, and the remainder's written ones), at least topk of them, and no
// larger logit is missing, so the selection over them is the selection over
// the row.
__global__ void __launch_bounds__(kNT, kTopkCtasPerSm) cand_select_kernel(CandTopkParams p)
{
    extern __shared__ __align__(16) unsigned char topk_smem_raw[];
    TopkSmem& sm = *reinterpret_cast<TopkSmem*>(topk_smem_raw);
    int buf = 0;
    const unsigned k = (unsigned)p.topk;
    for (int i = blockIdx.x; i < p.rows; i += gridDim.x) {
        int lo, hi;
        cand_range(p, i, lo, hi);
        const unsigned n = (unsigned)(hi - lo);
        int* out = p.indices + (long long)i * p.topk;
        const unsigned taken = n < k ? n : k;
        __syncthreads();   // the previous row's shared state is no longer read
        if (n <= k) {
            for (unsigned c = threadIdx.x; c < n; c += kNT)
                out[c] = lo + (int)c;
        } else {
            CandView cv;
            cv.vals = p.vals + (long long)i * p.ldo;
            cv.mask = p.mask + (long long)i * (p.ldo >> 5);
            cv.c_lo = lo;
            cv.c_hi = hi;
            cv.s = __ldg(p.rem_hi + i);
            cv.thr = __ldg(p.thr + i);
            auto walk = [&](auto&& f) { for_cand_row(cv, f); };
            // common case: the estimate t0 leaves between topk and kCap
            // candidates; one walk compacts them and the rest is in shared memory
            const unsigned t0 = __ldg(p.t0 + i);
            bool done = false;
            if (t0 != 0u) {
                const unsigned m = compact_walk(sm, walk, t0, buf);
                if (m >= k && m <= (unsigned)kCap) {
                    if (!select_from_list_rel(sm, m, k, t0, out, buf))
                        select_from_list(sm, m, k, out, buf);
                    done = true;
                }
            }
            if (!done) {
                clear_hist<kBins12>(sm);
                walk([&](const unsigned(&key)[kPer], unsigned okm, RowIdx) {
#pragma unroll
                    for (int e = 0; e < kPer; ++e)
                        if ((okm >> e) & 1u)
                            atomicAdd(&sm.hist[key[e] >> 20], 1u);
                });
                __syncthreads();
                unsigned b1, above1, n1;
                select_bin<kBins12>(sm, k, buf, b1, above1, n1);
                if (above1 + n1 <= (unsigned)kCap) {
                    const unsigned mm = compact_walk(sm, walk, b1 << 20, buf);
                    finish_row(
                        sm, [&](auto&& f) { for_cand(sm, mm < (unsigned)kCap ? mm : (unsigned)kCap, f); },
                        b1, above1, k, out, buf);
                } else {
                    finish_row(sm, walk, b1, above1, k, out, buf);
                }
            }
        }
        for (unsigned c = taken + threadIdx.x; c < k; c += kNT)
            out[c] = -1;
    }
}

// Sets the shared-memory limit of a selection kernel once per device.
template <class K>
cudaError_t set_topk_smem(K kern, std::atomic<unsigned long long>& attr_set)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (!(attr_set.load() & bit) || !bit) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(TopkSmem));
        if (e != cudaSuccess)
            return e;
        attr_set.fetch_or(bit);
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, int grid, cudaStream_t stream)
{
    const size_t smem = sizeof(TopkSmem);
    // per-device function attribute: set once on each device (see launch.h)
    static std::atomic<unsigned long long> attr_set{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (!(attr_set.load() & bit) || !bit) {
        e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set.fetch_or(bit);
    }
    topk_kernel<<<grid, kNT, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cand_split(const CandTopkParams& p, cudaStream_t stream)
{
    cand_split_kernel<<<(p.rows + 255) / 256, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cand_threshold(const CandTopkParams& p, int grid, cudaStream_t stream)
{
    static std::atomic<unsigned long long> attr_set{0};
    cudaError_t e = set_topk_smem(cand_threshold_kernel, attr_set);
    if (e != cudaSuccess)
        return e;
    cand_threshold_kernel<<<grid, kNT, sizeof(TopkSmem), stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cand_select(const CandTopkParams& p, int grid, cudaStream_t stream)
{
    static std::atomic<unsigned long long> attr_set{0};
    cudaError_t e = set_topk_smem(cand_select_kernel, attr_set);
    if (e != cudaSuccess)
        return e;
    cand_select_kernel<<<grid, kNT, sizeof(TopkSmem), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace mqa
