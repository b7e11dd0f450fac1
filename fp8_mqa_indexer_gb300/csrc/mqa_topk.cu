// mqa_topk.cu -- top-k key selection over rows of MQA logits.
//
// For each query row: the topk keys of the row's range with the largest
// logits, in ascending key order, padded with -1.  This is the `indices`
// input of the sparse-attention call on the "FlashMLA" page (parameters of
// flash_mla_with_kvcache: shape (batch, seq_len_q, topk), invalid entries
// -1).  Larger means later in the IEEE-754 totalOrder of the fp32 value;
// among equal values the smaller key is taken, so the result is unique.
//
// A persistent grid (two CTAs per SM) walks the rows, one row per CTA at a
// time.  Each logit maps to a 32-bit key whose unsigned order is totalOrder,
// and a radix select over three digits (bits 31..20, 19..8, 7..0) finds the
// k-th largest key T:
//   1. histogram of digit 1 over the row (the row's read from HBM) gives the
//      bin holding the k-th largest key;
//   2. every element in or above that bin is compacted, in key order, into
//      shared memory (a second read of the row, normally from L2);
//   3. histograms of digits 2 and 3 over the compacted elements of the bin
//      give T, the count of keys above T, and r = the number of keys equal to
//      T that are taken (the r smallest such keys);
//   4. one ordered pass over the compacted list writes each taken key at its
//      rank: (keys above T before it) + min(keys equal to T before it, r).
// If the bin and everything above it do not fit shared memory (many equal or
// nearly equal logits), steps 3 and 4 read the row from global memory.
// Rows with at most topk keys take every key without reading the logits.
#include "topk.h"

namespace mqa {
namespace {

constexpr int kNT = kTopkThreads;
constexpr int kNW = kNT / 32;
constexpr int kTile = 4 * kNT;   // elements per block-wide step (four per thread)
constexpr int kBins12 = 4096;    // digits 1 and 2
constexpr int kBins8 = 256;      // digit 3
constexpr int kCap = 8192;       // compacted elements held in shared memory

struct TopkSmem {
    unsigned hist[kBins12];
    unsigned cand_key[kCap];
    int cand_idx[kCap];
    unsigned warp_sum[2][kNW];
    unsigned sel_bin, sel_above, sel_count;
};

// Unsigned key whose order is the IEEE-754 totalOrder of v: negative values
// have every bit flipped, non-negative ones only the sign bit.
__device__ __forceinline__ unsigned order_key(float v)
{
    const unsigned u = __float_as_uint(v);
    return u ^ ((unsigned)((int)u >> 31) | 0x80000000u);
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

// The bin of hist[0, NBINS) that holds the need-th largest element (1 <= need
// <= the histogram's total): sel_bin, sel_above (elements in higher bins) and
// sel_count (elements in the bin).  Ends with the selection visible to all.
template <int NBINS>
__device__ __forceinline__ void select_bin(TopkSmem& sm, unsigned need, int& buf, unsigned& bin,
                                           unsigned& above, unsigned& count)
{
    constexpr int kPer = NBINS >= kNT ? NBINS / kNT : 1;
    const int b0 = threadIdx.x * kPer;
    unsigned h[kPer], s = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        h[q] = b0 + q < NBINS ? sm.hist[b0 + q] : 0u;
        s += h[q];
    }
    unsigned total;
    const unsigned before = block_exclusive_sum(s, sm.warp_sum[buf], total);
    buf ^= 1;
    unsigned acc = total - before - s;   // elements in the bins of higher threads
#pragma unroll
    for (int q = kPer - 1; q >= 0; --q) {
        if (acc < need && acc + h[q] >= need) {
            sm.sel_bin = (unsigned)(b0 + q);
            sm.sel_above = acc;
            sm.sel_count = h[q];
        }
        acc += h[q];
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

// f(key[4], idx[4], ok[4]) for each thread's four consecutive columns of
// every block-wide step over the range; all threads take the same number of
// steps, so f may synchronize the block.  Whole aligned groups load as one
// float4, the ragged ends element by element.
template <class F>
__device__ __forceinline__ void for_row(const RowView& r, F&& f)
{
    for (long long base = r.c_start; base < r.c_hi; base += kTile) {
        const long long c = base + 4 * threadIdx.x;
        float v[4];
        bool ok[4];
        if (c >= r.c_lo && c + 4 <= r.c_hi) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(r.ptr + c));
            v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
            ok[0] = ok[1] = ok[2] = ok[3] = true;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ok[e] = c + e >= r.c_lo && c + e < r.c_hi;
                v[e] = ok[e] ? __ldg(r.ptr + c + e) : 0.f;
            }
        }
        unsigned key[4];
        int idx[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            key[e] = order_key(v[e]);
            idx[e] = (int)(c + e) + r.key_of_col0;
        }
        f(key, idx, ok);
    }
}

// Digit-1 histogram with four block-wide steps per trip, so that each thread
// has four 16-byte loads in flight.
__device__ __forceinline__ void hist_digit1(TopkSmem& sm, const RowView& r)
{
    for (long long base = r.c_start; base < r.c_hi; base += 4 * kTile) {
        float v[4][4];
        bool ok[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const long long c = base + g * kTile + 4 * threadIdx.x;
            if (c >= r.c_lo && c + 4 <= r.c_hi) {
                const float4 x = __ldg(reinterpret_cast<const float4*>(r.ptr + c));
                v[g][0] = x.x, v[g][1] = x.y, v[g][2] = x.z, v[g][3] = x.w;
                ok[g][0] = ok[g][1] = ok[g][2] = ok[g][3] = true;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ok[g][e] = c + e >= r.c_lo && c + e < r.c_hi;
                    v[g][e] = ok[g][e] ? __ldg(r.ptr + c + e) : 0.f;
                }
            }
        }
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (ok[g][e])
                    atomicAdd(&sm.hist[order_key(v[g][e]) >> 20], 1u);
    }
}

// f(key[4], idx[4], ok[4]) over the first m compacted elements, four per
// thread per block-wide step, in key order.
template <class F>
__device__ __forceinline__ void for_cand(const TopkSmem& sm, unsigned m, F&& f)
{
    for (unsigned base = 0; base < m; base += kTile) {
        unsigned key[4];
        int idx[4];
        bool ok[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const unsigned k = base + 4 * threadIdx.x + e;
            ok[e] = k < m;
            key[e] = ok[e] ? sm.cand_key[k] : 0u;
            idx[e] = ok[e] ? sm.cand_idx[k] : 0;
        }
        f(key, idx, ok);
    }
}

template <int NBINS>
__device__ __forceinline__ void clear_hist(TopkSmem& sm)
{
    for (int b = threadIdx.x; b < NBINS; b += kNT)
        sm.hist[b] = 0u;
    __syncthreads();
}

// Digits 2 and 3 over `each` (a for_row or for_cand walk), then the ordered
// write of the selection.  b1 / above1 come from digit 1.
template <class Walk>
__device__ __forceinline__ void finish_row(TopkSmem& sm, Walk&& each, unsigned b1, unsigned above1,
                                           unsigned k, int* out, int& buf)
{
    clear_hist<kBins12>(sm);
    each([&](const unsigned(&key)[4], const int(&)[4], const bool(&ok)[4]) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (ok[e] && (key[e] >> 20) == b1)
                atomicAdd(&sm.hist[(key[e] >> 8) & 0xfffu], 1u);
    });
    __syncthreads();
    unsigned b2, above2, cnt;
    select_bin<kBins12>(sm, k - above1, buf, b2, above2, cnt);
    const unsigned prefix = (b1 << 12) | b2;
    clear_hist<kBins8>(sm);
    each([&](const unsigned(&key)[4], const int(&)[4], const bool(&ok)[4]) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (ok[e] && (key[e] >> 8) == prefix)
                atomicAdd(&sm.hist[key[e] & 0xffu], 1u);
    });
    __syncthreads();
    unsigned b3, above3;
    select_bin<kBins8>(sm, k - above1 - above2, buf, b3, above3, cnt);
    const unsigned T = (prefix << 8) | b3;
    const unsigned r = k - above1 - above2 - above3;   // keys equal to T that are taken
    unsigned gt_run = 0, eq_run = 0;
    each([&](const unsigned(&key)[4], const int(&idx)[4], const bool(&ok)[4]) {
        unsigned g = 0, q = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            g += ok[e] && key[e] > T;
            q += ok[e] && key[e] == T;
        }
        // a step holds at most kTile < 2^16 elements: both counts fit 16 bits
        unsigned tot;
        const unsigned off = block_exclusive_sum(g | (q << 16), sm.warp_sum[buf], tot);
        buf ^= 1;
        unsigned gb = gt_run + (off & 0xffffu), eb = eq_run + (off >> 16);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (!ok[e])
                continue;
            if (key[e] > T) {
                const unsigned pos = gb + min(eb, r);
                if (pos < k)
                    out[pos] = idx[e];
                ++gb;
            } else if (key[e] == T) {
                if (eb < r && gb + eb < k)
                    out[gb + eb] = idx[e];
                ++eb;
            }
        }
        gt_run += tot & 0xffffu;
        eq_run += tot >> 16;
    });
}

__global__ void __launch_bounds__(kNT, kTopkCtasPerSm) topk_kernel(TopkParams p)
{
    extern __shared__ __align__(16) unsigned char topk_smem_raw[];
    TopkSmem& sm = *reinterpret_cast<TopkSmem*>(topk_smem_raw);
    int buf = 0;
    const unsigned k = (unsigned)p.topk;
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
            // ---- digit 1 over the row
            clear_hist<kBins12>(sm);
            hist_digit1(sm, r);
            __syncthreads();
            unsigned b1, above1, n1;
            select_bin<kBins12>(sm, k, buf, b1, above1, n1);
            const unsigned m = above1 + n1;   // elements in bin b1 or above
            if (m <= (unsigned)kCap) {
                // ---- compact those elements, in key order, into shared memory
                unsigned run = 0;
                for_row(r, [&](const unsigned(&key)[4], const int(&idx)[4], const bool(&ok)[4]) {
                    bool f[4];
                    unsigned cnt = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        f[e] = ok[e] && (key[e] >> 20) >= b1;
                        cnt += f[e];
                    }
                    unsigned tot;
                    unsigned pos = run + block_exclusive_sum(cnt, sm.warp_sum[buf], tot);
                    buf ^= 1;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (f[e] && pos < (unsigned)kCap) {
                            sm.cand_key[pos] = key[e];
                            sm.cand_idx[pos] = idx[e];
                        }
                        pos += f[e];
                    }
                    run += tot;
                });
                __syncthreads();
                const unsigned mm = run < (unsigned)kCap ? run : (unsigned)kCap;
                finish_row(
                    sm, [&](auto&& f) { for_cand(sm, mm, f); }, b1, above1, k, out, buf);
            } else {
                finish_row(
                    sm, [&](auto&& f) { for_row(r, f); }, b1, above1, k, out, buf);
            }
        }
        for (unsigned c = taken + threadIdx.x; c < k; c += kNT)
            out[c] = -1;
    }
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, int grid, cudaStream_t stream)
{
    const size_t smem = sizeof(TopkSmem);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    topk_kernel<<<grid, kNT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace mqa
