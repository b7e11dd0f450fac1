// mqa_kernel.cuh -- the MQA logits kernel for sm_103a (dense and paged KV).
//
// What it computes ("How to Implement MQA (Multi-Query Attention) Logits
// Computation with DeepGEMM", section "Core Architecture Components"): for
// query token i and key j in its range,
//     logits[i, j] = sum_h w[i,h] * ReLU(s[j] * <q[i,h,:], kv[j,:]>)
// with E4M3 q/kv, fp32 per-key scale s and per-head weight w (fp32 or bf16),
// fp32 or bf16 output, and -inf outside the range in clean mode ("[PR #435]
// Improve SM100 MX MQA logits clean-output performance", section "Standalone
// performance reproducer").  MX instances take MXFP8 or MXFP4 q/kv with UE8M0
// block scales in place of s (same page, sections "Performance" and
// "Validation").
//
// Design (this library's own, for GB300):
//  * Keys sit on the MMA M dimension: one 128-key tile of kv is the A operand
//    (128 TMEM lanes = 128 keys) and a block of `tok` query tokens x H heads is
//    the B operand (N = tok * H <= 256 columns).  Both are K-major (D
//    contiguous) exactly as they lie in HBM, so TMA copies them unchanged into
//    swizzled shared memory and tcgen05.mma (kind::f8f6f4, E4M3 x E4M3 -> F32)
//    accumulates x[key, (token, head)] in TMEM.
//  * Epilogue threads each own one key (one TMEM lane) and reduce over heads in
//    registers: acc = sum_h w[h] * max(x, 0), then multiply by s[j] once (exact
//    rewrite of ReLU(s x) for s >= 0; a warp that sees a negative scale sums
//    w x and w |x| instead, since ReLU(y) = (y + |y|) / 2).  The head weights
//    stay in registers for a whole query block.  For a fixed token the 128
//    threads of a warp group write 128 consecutive floats: coalesced rows.
//  * One persistent CTA per SM walks a contiguous slice of the (query block,
//    key tile) work list: dense slices come from an in-kernel prefix sum over
//    the query blocks; paged slices come from the schedule written by
//    paged_mqa_logits_metadata.
//  * Warp roles (640 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
//    owner, warps 2-3 write -inf into the columns no tile covers (clean mode),
//    warps 4-19 are four epilogue warp groups of 64 columns each (groups
//    without columns in a launch leave at once).  Paged calls: warps 0 and 2
//    produce alternate units (page-id lookups and gathers), warp 3 alone fills.
//  * MX: the block scales go into TMEM with tcgen05.cp beside the two
//    accumulators (units of 192 columns) and the MMA is the block-scaled
//    kind::mxf8f6f4; dense calls transpose the key scales in the producer,
//    paged calls copy them by TMA with the pages and the MMA warp transposes.
//  * Candidate instances (output type CandOut) serve the fused logits + top-k
//    call: a logit of a row's range is kept only when it is not below the
//    row's threshold; the kept logits of each 32-key line are written packed
//    at the front of the line (zero-padded to a 32-byte boundary) with a
//    32-bit mask of their keys; nothing else is written (no -inf fill).
//  * Pipelines: a ring of key tiles (+ their scales and a small work record),
//    two query-block buffers (+ weights and per-token ranges) and two TMEM
//    accumulators of 256 columns; every hand-off is an mbarrier, every wait is
//    bounded (ptx.cuh, wait_bounded).
#pragma once
#include <cuda_bf16.h>

#include <climits>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace mqa {

constexpr int kBlockKV = 128;      // keys per tile == MMA M == TMEM lanes
constexpr int kMaxN = 256;         // TMEM columns per accumulator buffer
// Thread layout: warp group 0 holds the producer, MMA and fill warps; the
// epilogue warp groups split the 256 accumulator columns.  kEpiCols picks the
// split: 64 columns (four epilogue groups, 640 threads) or 128 (two groups,
// 384 threads).  The register budget follows from the thread count.
constexpr int kEpiCols = 64;                          // accumulator columns per epilogue group
constexpr int kNumEpiWarps = 4 * (kMaxN / kEpiCols);
constexpr int kEpiWarp0 = 4;                          // epilogue warps follow warp group 0
constexpr int kThreads = 32 * (kEpiWarp0 + kNumEpiWarps);
constexpr int kLaunchRegs = (65536 / kThreads) & ~7;  // registers per thread at launch
constexpr int kRegsCtl = (kEpiCols == 64) ? 32 : 56;  // warp group 0 after the split
constexpr int kRegsEpi = (kEpiCols == 64) ? 112 : 216;
constexpr int kPiece = (kEpiCols == 64) ? 16 : 32;    // accumulator columns per TMEM load
constexpr int kMaxTokW = kEpiCols / 8;                // tokens in one group's columns (H >= 8)
static_assert(128 * kRegsCtl + 32 * kNumEpiWarps * kRegsEpi <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");

enum : unsigned { kFlagClean = 1u, kFlagCompressed = 2u };
enum : int { kFirstOfBlock = 1, kLastOfBlock = 2 };

struct UnitInfo {
    int b;        // query block (dense) or sequence (paged)
    int t;        // key tile: keys [t*128, t*128+128)
    int qbuf;     // which query-block buffer holds block b
    int flags;    // kFirstOfBlock | kLastOfBlock (within this CTA's slice)
};

// Output row of one query token: where its logits go and which keys are valid.
// The logits of keys j in [slo, shi) go to logits[off + j]; keys in
// [vlo, vhi) get their value, the rest of that window -inf (clean mode).  In
// compressed mode off is shifted by the row's first key; a row that does not
// exist has an empty window.
struct __align__(16) TokRow {
    int slo, shi;    // keys stored
    int vlo, vhi;    // keys with a value
    long long off;   // offset of key 0 of the row in the logits
    long long pad;   // candidate instances: the row's threshold (fp32 bits, low half)
};

// Output type of the candidate instances: per 32-key line, the kept fp32
// logits packed at the front of the line and a mask of their keys.
struct CandOut {};

struct Params {
    void* logits;            // float, or __nv_bfloat16 (bf16 instances); candidates: float
    long long ldo;
    unsigned flags;
    // dense
    int S_q;
    int S_kv;
    const int* k_start;
    const int* k_end;
    const float* kv_scale;   // dense: scanned once for negative scales
    // paged
    const int* context_lens;
    const int* block_table;
    const int* schedule_meta;
    int B;
    int next_n;
    int block_kv;
    int max_blocks;
    int num_blocks;          // physical blocks of the pool (bounds the scale-word loads)
    int kv_page_rows;        // paged: rows of D bytes from one page's keys to the next's
    // shared
    long long width;     // logical columns of an uncompressed row
    int width_i;         // the same, as an int (below 2^31 - 256)
    int tok;             // query tokens per work unit
    int tok0;            // paged: first token (within its sequence) of this launch's query atom
    int blk_stride;      // output rows between query blocks: tok (dense) or next_n (paged)
    int num_q_blocks;    // dense: ceil(S_q / tok); paged: B
    int rows;            // output rows: S_q or B * next_n
    // MX (block-scaled) dense calls: UE8M0 scales, four per int32, byte b for
    // elements [32 b, 32 b + 32) of a row
    const uint32_t* q_sf;    // [S_q * H]
    const uint32_t* kv_sf;   // [S_kv]
    uint32_t mx_fmt;         // element format of q and kv: kFmtE4M3 or kFmtE2M1
    int w_bf16;              // weights are bf16 (else fp32)
    // candidate instances: row r, line L (keys [32 L, 32 L + 32)) has its mask
    // at cand_mask[r * ldo / 32 + L] (row `rows` is scratch for the absent
    // rows of a last query block; ldo is a multiple of 128); a logit v of the
    // row's range is kept unless v < cand_thr[r] (all of them when cand_thr is
    // null)
    unsigned* cand_mask;
    const float* cand_thr;
    long long wait_limit;
    unsigned* status;
};

template <int D>
struct Cfg {
    static constexpr int kStages = (D == 128) ? 8 : 12;
    static constexpr int kKVTileBytes = kBlockKV * D;
    static constexpr int kQTileBytes = kMaxN * D;
};

// MX calls: accumulator columns of a unit (three tokens at H = 64), so that the
// two 256-column buffers leave room in TMEM for the scale factors, which sit
// at columns kMxSfCol.. of the first buffer's unused tail: SFA in two slots of
// four columns (by unit parity), SFB in two slots of eight (by query buffer).
constexpr int kMxN = 192;
constexpr int kMxSfaCol = kMxN;          // 192..199
constexpr int kMxSfbCol = kMxN + 8;      // 200..215

template <int D, bool MX = false>
struct __align__(1024) Smem {
    uint8_t q[2][Cfg<D>::kQTileBytes];
    uint8_t kv[Cfg<D>::kStages][Cfg<D>::kKVTileBytes];
    float scale[Cfg<D>::kStages][kBlockKV];
    float w[2][kMaxN];
    int2 range[2][32];
    UnitInfo info[Cfg<D>::kStages];
    uint64_t full[Cfg<D>::kStages];
    uint64_t empty[Cfg<D>::kStages];
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t mma_done;
    uint64_t neg_bar;        // dense: the epilogue warps' scale scan is done
    uint32_t tmem_base;
    int abort_flag;
    int any_neg;             // dense: some key scale is negative
    int start_b;
    int start_t;
    int n_units;
    long long scan[kThreads / 32];
    TokRow tokrow[kNumEpiWarps][kMaxTokW];   // per epilogue warp: its tokens' rows
    // MX: scale factors laid out for tcgen05.cp (32 rows x 16 bytes, row r
    // word j = the scales of matrix row 32 j + r): per key-tile stage (A =
    // keys) and per query buffer, in two halves of 128 rows (B = token x head)
    alignas(16) uint32_t sfa[MX ? Cfg<D>::kStages : 1][32][4];
    alignas(16) uint32_t sfb[MX ? 2 : 1][2][32][4];
};

// ----------------------------------------------------------------- ranges
// Dense range of row i, intersected with [0, S_kv): returns [lo, hi), lo <= hi.
__device__ __forceinline__ int2 dense_range(const Params& p, int i)
{
    int lo = min(max(__ldg(p.k_start + i), 0), p.S_kv);
    int hi = min(max(__ldg(p.k_end + i), lo), p.S_kv);
    return make_int2(lo, hi);
}

// Paged range of token t (0 <= t < next_n) of a sequence with context ctx:
// [0, ctx - next_n + t + 1) intersected with [0, width).
__device__ __forceinline__ int2 paged_range(const Params& p, int ctx, int t)
{
    long long hi = (long long)ctx - p.next_n + t + 1;
    hi = hi < 0 ? 0 : (hi > p.width ? p.width : hi);
    return make_int2(0, (int)hi);
}

__device__ __forceinline__ int paged_tiles(int ctx)
{
    return ctx > 0 ? (ctx + kBlockKV - 1) / kBlockKV : 0;
}

// Key tiles [tlo, thi) touched by dense query block b (one thread).
__device__ __forceinline__ void dense_block_tiles(const Params& p, int b, int& tlo, int& thi)
{
    const int r0 = b * p.tok;
    const int r1 = min(r0 + p.tok, p.S_q);
    int mn = INT_MAX, mx = 0;
    for (int i = r0; i < r1; ++i) {
        int2 r = dense_range(p, i);
        if (r.y > r.x) {
            mn = min(mn, r.x);
            mx = max(mx, r.y);
        }
    }
    if (mx == 0) {
        tlo = thi = 0;
    } else {
        tlo = mn / kBlockKV;
        thi = (mx + kBlockKV - 1) / kBlockKV;
    }
}

// Same, cooperatively by a full warp (tok <= 32); lane k also returns token
// k's range in `mine`.
__device__ __forceinline__ void dense_block_tiles_warp(const Params& p, int b, int lane, int& tlo,
                                                       int& thi, int2& mine)
{
    const int i = b * p.tok + lane;
    int2 r = make_int2(0, 0);
    if (lane < p.tok && i < p.S_q)
        r = dense_range(p, i);
    mine = r;
    const bool ne = r.y > r.x;
    const int mn = __reduce_min_sync(0xffffffffu, ne ? r.x : INT_MAX);
    const int mx = __reduce_max_sync(0xffffffffu, ne ? r.y : 0);
    if (mx == 0) {
        tlo = thi = 0;
    } else {
        tlo = mn / kBlockKV;
        thi = (mx + kBlockKV - 1) / kBlockKV;
    }
}

__device__ __forceinline__ long long block_units(const Params& p, bool paged, int b)
{
    if (paged)
        return paged_tiles(__ldg(p.context_lens + b));
    int tlo, thi;
    dense_block_tiles(p, b, tlo, thi);
    return thi - tlo;
}

// -------------------------------------------------------- -inf fill of rows
// -inf of the output element type (fp32 0xff800000, bf16 0xff80).
template <typename OutT> __device__ __forceinline__ OutT neg_inf();
template <> __device__ __forceinline__ float neg_inf<float>() { return __int_as_float(0xff800000u); }
template <> __device__ __forceinline__ __nv_bfloat16 neg_inf<__nv_bfloat16>()
{
    return __ushort_as_bfloat16((unsigned short)0xff80u);
}

template <typename OutT> __device__ __forceinline__ OutT to_out(float v);
template <> __device__ __forceinline__ float to_out<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}

// Writes -inf to row[c0, c1) with one warp: scalar head to a 16-byte boundary,
// 16-byte body, scalar tail.
template <typename OutT>
__device__ __forceinline__ void warp_fill_neg_inf(OutT* row, long long c0, long long c1, int lane)
{
    if (c0 >= c1)
        return;
    constexpr int kVec = 16 / sizeof(OutT);   // elements per 16-byte store
    const OutT ninf = neg_inf<OutT>();
    const long long mis =
        (long long)((reinterpret_cast<uintptr_t>(row + c0) / sizeof(OutT)) & (kVec - 1));
    const long long head = min((kVec - mis) & (kVec - 1), c1 - c0);
    if (lane < head)
        row[c0 + lane] = ninf;
    long long a = c0 + head;
    const long long nvec = (c1 - a) / kVec;
    uint4* v = reinterpret_cast<uint4*>(row + a);
    const uint32_t w = sizeof(OutT) == 4 ? 0xff800000u : 0xff80ff80u;   // -inf, packed
    const uint4 f4 = make_uint4(w, w, w, w);
    for (long long k = lane; k < nvec; k += 32)
        v[k] = f4;
    a += nvec * kVec;
    for (long long c = a + lane; c < c1; c += 32)
        row[c] = ninf;
}

// A bounded wait taken by a whole warp: every lane gets the same answer, so a
// timeout never splits the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                          unsigned sleep_ns = 0)
{
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, w, sleep_ns));
}

// Back-off of waiters off the critical path (ns between polls).
constexpr unsigned kProducerSleepNs = 256;
constexpr unsigned kMmaSleepNs = 0;

// --------------------------------------------------------------- epilogue
// Epilogue of one warp: per work unit it reads its 32 keys x 64 columns of
// the TMEM accumulator (keys on lanes, (token, head) on columns) in pieces of
// 16 columns, reduces sum_h w[h] * ReLU(s x) per token and writes the
// row-masked logits.  The 64 head weights of its columns stay in registers
// for the whole query block; the output row and key range of each of its
// tokens sit in shared memory, written once per block.  The accumulator goes
// back to the MMA warp as soon as the last piece is in registers.
//
// Arithmetic per element: with s >= 0 for every key of the warp, ReLU(s x) =
// s * max(x, 0), so the warp accumulates w * max(x, 0) with packed FFMA2 and
// scales once per token.  A warp that holds a negative scale uses
// ReLU(y) = (y + |y|) / 2 instead: it accumulates A = sum w x and
// B = sum w |x| and forms (s A + |s| B) / 2, which equals sum w ReLU(s x) for
// either sign of s.
template <int H, int D, bool MX = false, typename OutT = float>
struct Epilogue {
    static_assert(H >= 8 && H <= kEpiCols, "a warp's columns must hold whole tokens");
    using C = Cfg<D>;
    static constexpr int S = C::kStages;
    static constexpr int kTokW = kEpiCols / H;   // tokens in a warp's columns
    static constexpr bool kCand = std::is_same<OutT, CandOut>::value;
    static_assert(kTokW <= kMaxTokW, "token rows do not fit the shared table");

    struct Unit {
        int buf;
        UnitInfo info;
        float s;
    };

    Smem<D, MX>& sm;
    const Params& p;
    const WaitCtx& wctx;
    uint32_t tmem_lane;   // TMEM address of this warp's lanes and first column
    int n_units;
    int row;              // key row of this thread within the tile (TMEM lane)
    int col0;             // first accumulator column of this warp
    int tok0;             // first token of those columns within the query block
    int ntok;             // tokens of the block that fall in those columns
    int slot;             // this warp's index among the epilogue warps
    float2 w2[kEpiCols / 2];

    __device__ __forceinline__ void enter_block(const UnitInfo& info)
    {
        if (p.w_bf16) {
            // bf16 weights, widened exactly: a bf16 is the top half of an fp32
            const uint4* w8 = reinterpret_cast<const uint4*>(
                reinterpret_cast<const uint16_t*>(&sm.w[info.qbuf][0]) + col0);
#pragma unroll
            for (int i = 0; i < kEpiCols / 8; ++i) {
                const uint4 v = w8[i];
                const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    w2[4 * i + j] = make_float2(__uint_as_float(x[j] << 16),
                                                __uint_as_float(x[j] & 0xffff0000u));
            }
        } else {
            const float4* w4 = reinterpret_cast<const float4*>(&sm.w[info.qbuf][col0]);
#pragma unroll
            for (int i = 0; i < kEpiCols / 4; ++i) {
                const float4 v = w4[i];
                w2[2 * i] = make_float2(v.x, v.y);
                w2[2 * i + 1] = make_float2(v.z, v.w);
            }
        }
        const int a = threadIdx.x & 31;
        __syncwarp();
        if (a < kTokW) {
            TokRow t;
            const int r = info.b * p.blk_stride + p.tok0 + tok0 + a;
            const int2 rg = sm.range[info.qbuf][tok0 + a];   // within [0, width)
            t.slo = t.shi = t.vlo = t.vhi = 0;
            t.off = kCand ? (long long)p.rows * p.ldo : 0;   // candidates: the scratch row
            t.pad = 0;
            if (a < ntok && r < p.rows) {
                t.off = (long long)r * p.ldo;
                if (kCand)
                    t.pad = (long long)__float_as_uint(p.cand_thr ? __ldg(p.cand_thr + r)
                                                                  : __int_as_float(0xff800000));
                t.slo = t.vlo = rg.x;
                t.shi = t.vhi = rg.y;
                if (p.flags & kFlagCompressed) {   // column j - lo, below ldo
                    t.off -= rg.x;
                    if ((long long)rg.x + p.ldo < rg.y)
                        t.shi = t.vhi = (int)(rg.x + p.ldo);
                } else if (p.flags & kFlagClean) {   // -inf outside the range
                    t.slo = 0;
                    t.shi = p.width_i;
                }
            }
            sm.tokrow[slot][a] = t;
        }
        __syncwarp();
    }

    // Waits for unit v's inputs and accumulator; hands the key-tile stage back
    // to the producer (its scale and work record have been read).
    __device__ __forceinline__ bool begin(int stage, uint32_t phase, int v, int& k_block, Unit& st)
    {
        if (!warp_wait_fast(smem_u32(&sm.full[stage]), phase, wctx))
            return false;
        st.info = sm.info[stage];
        // MX: the block scales are applied inside the MMA; no per-key scale
        st.s = MX ? 1.f : sm.scale[stage][row];
        if (st.info.flags & kFirstOfBlock) {
            ++k_block;
            if (!warp_wait_fast(smem_u32(&sm.q_full[st.info.qbuf]), (k_block >> 1) & 1, wctx))
                return false;
            enter_block(st.info);
        }
        __syncwarp();
        mbar_arrive_one_per_warp(smem_u32(&sm.empty[stage]));
        st.buf = v & 1;
        if (!warp_wait_fast(smem_u32(&sm.acc_full[st.buf]), (v >> 1) & 1, wctx))
            return false;
        tc_fence_after();
        return true;
    }

    __device__ __forceinline__ void release(const Unit& st)
    {
        tc_fence_before();
        __syncwarp();
        mbar_arrive_one_per_warp(smem_u32(&sm.acc_empty[st.buf]));
    }

    __device__ __forceinline__ void finish(const Unit& st)
    {
        if (st.info.flags & kLastOfBlock) {
            __syncwarp();
            mbar_arrive_one_per_warp(smem_u32(&sm.q_empty[st.info.qbuf]));
        }
    }

    // Mask and store one logit of a token row.
    __device__ __forceinline__ void store(const Unit& st, const TokRow& t, float v)
    {
        // key index; the host keeps widths below 2^31 - 256 so this fits an int
        const int j = st.info.t * kBlockKV + row;
        if constexpr (kCand) {
            // The warp's 32 lanes are the 32 keys of one line (row = 32 quad +
            // lane): one ballot gives the line's mask and each kept logit's
            // place.  "not below" keeps NaNs: a superset of the keys at or
            // above the threshold's order key is all the selection needs.
            const bool take =
                j >= t.vlo && j < t.vhi && !(v < __uint_as_float((unsigned)t.pad));
            const unsigned m = __ballot_sync(0xffffffffu, take);
            const int lane = row & 31;
            const int cnt = __popc(m);
            float* line = static_cast<float*>(p.logits) + t.off + (j - lane);
            if (take)   // packed at the front of the line, in key order
                line[__popc(m & ((1u << lane) - 1u))] = v;
            // zeros up to the next 32-byte boundary: whole sectors only, so no
            // partly written sector is filled from DRAM
            if (lane >= cnt && lane < ((cnt + 7) & ~7))
                line[lane] = 0.f;
            // every line of the tile gets a mask (a row's masks are read only
            // over the range this launch covers for it)
            if (lane == 0)
                p.cand_mask[(t.off >> 5) + ((j - lane) >> 5)] = m;
        } else {
            // one predicated store: the logit, -inf (clean) or nothing
            if (j >= t.slo && j < t.shi)
                static_cast<OutT*>(p.logits)[t.off + j] =
                    (j >= t.vlo && j < t.vhi) ? to_out<OutT>(v) : neg_inf<OutT>();
        }
    }

    // Columns [c0, c0 + P) of the warp's slice, already in x.
    template <bool POS, int P>
    __device__ __forceinline__ void piece_math(const Unit& st, int c0, const float (&x)[P],
                                               float2& a0, float2& a1, float2& b0)
    {
#pragma unroll
        for (int k = 0; k < P; k += 4) {
            const int c = c0 + k;
            const float2 wa = w2[c >> 1], wb = w2[(c >> 1) + 1];
            if constexpr (POS) {
                a0 = __ffma2_rn(wa, make_float2(fmaxf(x[k], 0.f), fmaxf(x[k + 1], 0.f)), a0);
                a1 = __ffma2_rn(wb, make_float2(fmaxf(x[k + 2], 0.f), fmaxf(x[k + 3], 0.f)), a1);
            } else {
                a0 = __ffma2_rn(wa, make_float2(x[k], x[k + 1]), a0);
                b0 = __ffma2_rn(wa, make_float2(fabsf(x[k]), fabsf(x[k + 1])), b0);
                a0 = __ffma2_rn(wb, make_float2(x[k + 2], x[k + 3]), a0);
                b0 = __ffma2_rn(wb, make_float2(fabsf(x[k + 2]), fabsf(x[k + 3])), b0);
            }
            if ((c + 4) % H == 0) {   // last columns of token c / H
                float v;
                if constexpr (POS) {
                    const float2 t = __fadd2_rn(a0, a1);
                    v = MX ? t.x + t.y : st.s * (t.x + t.y);
                } else {
                    v = 0.5f * fmaf(st.s, a0.x + a0.y, fabsf(st.s) * (b0.x + b0.y));
                }
                store(st, sm.tokrow[slot][c / H], v);
                a0 = a1 = b0 = make_float2(0.f, 0.f);
            }
        }
    }

    // Load and wait as two statements: the compiler may schedule the previous
    // piece's arithmetic between them, which hides the TMEM latency.
    template <int P>
    __device__ __forceinline__ void load(uint32_t taddr, float (&x)[P])
    {
        static_assert(P == 16 || P == 32, "TMEM pieces are 16 or 32 columns");
        tmem_ld_async<P>(taddr, x);
        tmem_wait<P>(x);
    }

    // One unit over the first NC columns of the warp's slice (the columns that
    // hold tokens of the block, rounded up to a power of two >= 16), read in
    // pieces of kPiece columns, double-buffered: the next piece is in flight
    // while the current one is reduced.  POS: every scale of the warp is >= 0.
    template <bool POS, int NC>
    __device__ __forceinline__ void reduce(const Unit& st)
    {
        constexpr int P = NC < kPiece ? NC : kPiece;
        const uint32_t taddr = tmem_lane + (uint32_t)(st.buf * kMaxN);
        float2 a0 = make_float2(0.f, 0.f), a1 = a0, b0 = a0;
        constexpr int NP = NC / P;
        float xa[P], xb[P];
        tmem_ld_async<P>(taddr, xa);
        tmem_wait<P>(xa);
#pragma unroll
        for (int pc = 0; pc < NP; ++pc) {
            float(&cur)[P] = (pc & 1) ? xb : xa;
            float(&nxt)[P] = (pc & 1) ? xa : xb;
            if (pc + 1 < NP)
                tmem_ld_async<P>(taddr + P * (pc + 1), nxt);
            else
                release(st);
            piece_math<POS, P>(st, P * pc, cur, a0, a1, b0);
            if (pc + 1 < NP)
                tmem_wait<P>(nxt);
        }
    }

    // MIXED: some key scale may be negative, so each unit votes on its signs.
    template <int NC, bool MIXED>
    __device__ __forceinline__ void run()
    {
        int stage = 0;
        uint32_t phase = 0;
        int k_block = -1;
        // Eight units per trip (four below 64 heads, where a warp's columns
        // hold several tokens and the longer body runs out of instruction
        // cache): the accumulator buffer of each (and, with eight key-tile
        // stages, the stage too) is then known at compile time, the loop's
        // bookkeeping is shared, and the compiler can schedule one unit's tail
        // against the next unit's hand-offs.
        auto one = [&](int u) -> bool {
            Unit st;
            if (!begin(stage, phase, u, k_block, st))
                return false;
            if (!MIXED || __all_sync(0xffffffffu, st.s >= 0.f))
                reduce<true, NC>(st);
            else
                reduce<false, NC>(st);
            finish(st);
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
            return true;
        };
        int u = 0;
        if constexpr (H >= 64) {
            for (; u + 7 < n_units; u += 8) {
                if (!one(u) || !one(u + 1) || !one(u + 2) || !one(u + 3) || !one(u + 4) ||
                    !one(u + 5) || !one(u + 6) || !one(u + 7))
                    return;
            }
        } else {
            for (; u + 3 < n_units; u += 4) {
                if (!one(u) || !one(u + 1) || !one(u + 2) || !one(u + 3))
                    return;
            }
        }
        for (; u < n_units; ++u)
            if (!one(u))
                return;
    }
};

// ------------------------------------------------------------------ kernel
// MX = true: MXFP8 dense call (block-scaled E4M3 MMA, no per-key fp32 scale).
// OutT: float or __nv_bfloat16 logits (each fp32 logit rounded to nearest even).
template <int H, int D, bool PAGED, bool MX = false, typename OutT = float>
__global__ void __launch_bounds__(kThreads, 1)
    mqa_logits_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_kv,
                      const __grid_constant__ CUtensorMap tm_scale,
                      const __grid_constant__ CUtensorMap tm_w, const Params p)
{
    using C = Cfg<D>;
    constexpr int S = C::kStages;
    // Register split after set-up (launch: 640 threads x 96 = 61440): the
    // control warp group (producer, MMA, fill) gives registers to the four
    // epilogue warp groups, which hold a 64-column TMEM slice each;
    // 128 * ctl + 512 * epi <= 61440.
    static_assert(H >= 8 && H <= 128 && (H & (H - 1)) == 0, "H must be a power of two in [8,128]");
    static_assert(D == 64 || D == 128, "D must be 64 or 128");

    // Align the dynamic shared memory to 1024 B (the 128-byte swizzle repeat)
    // by pointer arithmetic on the shared array itself, so every access
    // through `sm` stays a shared-memory access (no generic addressing).
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    Smem<D, MX>& sm = *reinterpret_cast<Smem<D, MX>*>(smem_raw + pad);
    static_assert(!MX || D == 128, "MX calls have D = 128");

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    const int N = p.tok * H;

    // Epilogue warps whose columns hold tokens: the groups of the first N
    // columns.  The others (a paged unit narrower than 256 columns) leave at
    // once and take no part in any hand-off.
    const int n_epi = 4 * min(kNumEpiWarps / 4, (N + kEpiCols - 1) / kEpiCols);

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1 + n_epi);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(smem_u32(&sm.q_full[k]), 1);
            mbar_init(smem_u32(&sm.q_empty[k]), 1 + n_epi);
            mbar_init(smem_u32(&sm.acc_full[k]), 1);
            mbar_init(smem_u32(&sm.acc_empty[k]), n_epi);
        }
        mbar_init(smem_u32(&sm.mma_done), 1);
        mbar_init(smem_u32(&sm.neg_bar), kNumEpiWarps);
        sm.abort_flag = 0;
        sm.any_neg = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_kv);
        tma_prefetch_desc(&tm_scale);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), 512);
        tmem_relinquish();
    }
    // Calls are launched as programmatic dependents of the preceding kernel in
    // the stream (for the paged and the scheduled dense call, the schedule
    // kernel): the set-up above (shared memory and TMEM only) overlaps its
    // tail; every global access below comes after it has finished.
    grid_dependency_wait();

    // Work slice of this CTA: start (block, tile) and number of units.
    if (!PAGED && p.schedule_meta) {
        // dense, scheduled: entries cta and cta + 1 of the schedule written by
        // mqa_logits_metadata bound the slice; count its units over the
        // blocks it spans (the blocks' tile spans are recomputed here)
        const int NB = p.num_q_blocks;
        const int b0 = __ldg(p.schedule_meta + 2 * cta);
        const int t0 = __ldg(p.schedule_meta + 2 * cta + 1);
        const int b1 = __ldg(p.schedule_meta + 2 * cta + 2);
        const int t1 = __ldg(p.schedule_meta + 2 * cta + 3);
        bool ok = b0 >= 0 && b0 <= b1 && b1 <= NB && (b0 < NB || t0 == 0) && (b1 < NB || t1 == 0) &&
                  (b0 < b1 || t0 <= t1);
        long long local = 0;
        int bad = 0;
        if (ok) {
            for (int b = b0 + tid; b <= b1 && b < NB; b += kThreads) {
                int tlo, thi;
                dense_block_tiles(p, b, tlo, thi);
                const int lo = (b == b0) ? t0 : tlo;
                const int hi = (b == b1) ? t1 : thi;
                if (lo < tlo || hi > thi || lo > hi)   // the slice leaves the block's span
                    bad = 1;
                local += hi > lo ? hi - lo : 0;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            local += __shfl_xor_sync(0xffffffffu, local, o);
        if (lane == 0)
            sm.scan[warp] = local;
        ok = !__syncthreads_or(!ok || bad);
        if (tid == 0) {
            if (!ok)
                atomicOr(p.status, kDevErrBadSchedule);
            long long n = 0;
            for (int k = 0; k < kThreads / 32; ++k)
                n += sm.scan[k];
            sm.n_units = ok ? (int)n : 0;
            sm.start_b = b0;
            sm.start_t = t0;
        }
    } else if (!PAGED) {
        // Prefix sum of per-block tile counts over all threads, then locate
        // units [cta*U/G, (cta+1)*U/G).
        const int NB = p.num_q_blocks;
        const int chunk = (NB + kThreads - 1) / kThreads;
        const int b_lo = min(tid * chunk, NB);
        const int b_hi = min(b_lo + chunk, NB);
        long long local = 0;
        for (int b = b_lo; b < b_hi; ++b)
            local += block_units(p, false, b);
        long long incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        if (lane == 31)
            sm.scan[warp] = incl;
        __syncthreads();
        long long before = 0, total = 0;
        for (int k = 0; k < kThreads / 32; ++k) {
            if (k < warp)
                before += sm.scan[k];
            total += sm.scan[k];
        }
        const long long excl = before + incl - local;
        const long long u0 = (long long)cta * total / G;
        const long long u1 = (long long)(cta + 1) * total / G;
        if (tid == 0)
            sm.n_units = (int)(u1 - u0);
        if (u0 < u1 && u0 >= excl && u0 < excl + local) {
            long long acc = excl;
            for (int b = b_lo; b < b_hi; ++b) {
                int tlo, thi;
                dense_block_tiles(p, b, tlo, thi);
                if (u0 < acc + (thi - tlo)) {
                    sm.start_b = b;
                    sm.start_t = tlo + (int)(u0 - acc);
                    break;
                }
                acc += thi - tlo;
            }
        }
    } else {
        const int b0 = __ldg(p.schedule_meta + 2 * cta);
        const int t0 = __ldg(p.schedule_meta + 2 * cta + 1);
        const int b1 = __ldg(p.schedule_meta + 2 * cta + 2);
        const int t1 = __ldg(p.schedule_meta + 2 * cta + 3);
        bool ok = b0 >= 0 && b0 <= b1 && b1 <= p.B && t0 >= 0 && t1 >= 0;
        if (ok)
            ok = (b0 < p.B ? t0 <= paged_tiles(__ldg(p.context_lens + b0)) : t0 == 0) &&
                 (b1 < p.B ? t1 <= paged_tiles(__ldg(p.context_lens + b1)) : t1 == 0) &&
                 (b0 < b1 || t0 <= t1);
        if (!ok && tid == 0)
            atomicOr(p.status, kDevErrBadSchedule);
        long long local = 0;
        if (ok)
            for (int b = b0 + tid; b < b1; b += kThreads)
                local += paged_tiles(__ldg(p.context_lens + b));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            local += __shfl_xor_sync(0xffffffffu, local, o);
        if (lane == 0)
            sm.scan[warp] = local;
        __syncthreads();
        if (tid == 0) {
            long long tot = 0;
            for (int k = 0; k < kThreads / 32; ++k)
                tot += sm.scan[k];
            long long n = ok ? tot - t0 + t1 : 0;
            sm.n_units = (int)(n > 0 ? n : 0);
            sm.start_b = b0;
            sm.start_t = t0;
        }
    }
    // Candidate instances scan the key scales here, with every thread (in
    // their epilogue the scan measured slower: its registers crowd the
    // candidate store); the other dense instances scan in the epilogue warps.
    constexpr bool kScanFirst = !PAGED && !MX && std::is_same<OutT, CandOut>::value;
    int neg_first = 0;
    if constexpr (kScanFirst) {
        const int n4 = p.S_kv >> 2;
        const float4* s4 = reinterpret_cast<const float4*>(p.kv_scale);
        for (int k = tid; k < n4; k += kThreads) {
            const float4 v = __ldg(s4 + k);
            neg_first |= (v.x < 0.f) | (v.y < 0.f) | (v.z < 0.f) | (v.w < 0.f);
        }
        for (int k = (n4 << 2) + tid; k < p.S_kv; k += kThreads)
            neg_first |= __ldg(p.kv_scale + k) < 0.f;
    }
    neg_first = __syncthreads_or(neg_first);
    tc_fence_after();

    const uint32_t tmem_base = sm.tmem_base;
    const int n_units = sm.n_units;
    WaitCtx wctx{&sm.abort_flag, p.status, p.wait_limit};

    // Paged calls have two producer warps (0 and 2), each issuing the copies of
    // every other unit: a unit's page-id lookups and four copy requests keep
    // one warp busy longer than the rest of the pipeline needs per unit.
    constexpr int kProducers = PAGED ? 2 : 1;
    if (warp == 0 || (PAGED && warp == 2)) {
        // ================================================= TMA producer
        regs_dec<kRegsCtl>();
        const int pid = warp == 0 ? 0 : 1;   // units u with u % kProducers == pid are this warp's
        int b = sm.start_b;
        int t = sm.start_t;
        int k_block = 0;
        int tlo = 0, thi = 0;
        int2 myrange = make_int2(0, 0);
        int ctx = 0;
        // page-id window (paged): lane L holds the physical block of logical
        // pages wbase+L (win0) and wbase+32+L (win1, prefetched).
        int wbase = 0, win0 = -1, win1 = -1, npages = 0;
        const int ppt = PAGED ? kBlockKV / p.block_kv : 1;
        // bytes a copy of one D-element row counts on its barrier: MXFP4 rows
        // count their packed global bytes (D / 2), though each lands as D
        // bytes of shared memory
        auto elem_bytes = [&](int d) -> int { return MX && p.mx_fmt == kFmtE2M1 ? d / 2 : d; };
        auto page_id = [&](int pg) -> int {
            return (pg >= 0 && pg < npages)
                       ? __ldg(p.block_table + (long long)b * p.max_blocks + pg)
                       : -1;
        };
        auto enter_block = [&]() {
            if (PAGED) {
                ctx = b < p.B ? max(__ldg(p.context_lens + b), 0) : 0;
                tlo = 0;
                thi = paged_tiles(ctx);
                myrange = (lane < p.tok) ? paged_range(p, ctx, p.tok0 + lane) : make_int2(0, 0);
                npages = min((int)((min((long long)ctx, p.width) + p.block_kv - 1) / p.block_kv),
                             p.max_blocks);
                wbase = (t * ppt) & ~31;
                win0 = page_id(wbase + lane);
                win1 = page_id(wbase + 32 + lane);
            } else {
                dense_block_tiles_warp(p, b, lane, tlo, thi, myrange);
            }
        };
        if (n_units > 0)
            enter_block();
        bool first = true;
        int u_end = 0;
        int q_blk[2] = {-1, -1};   // the last two query blocks whose copies this warp issued
        for (int u = 0; u < n_units; ++u) {
            u_end = u;
            const bool mine = u % kProducers == pid;
            if (first && mine) {
                const int qb = k_block & 1;
                if (!warp_wait(smem_u32(&sm.q_empty[qb]), ((k_block >> 1) & 1) ^ 1, wctx,
                               kProducerSleepNs))
                    break;
                if (lane < p.tok)
                    sm.range[qb][lane] = myrange;
                if constexpr (MX) {
                    // the block's B-operand scales, transposed for tcgen05.cp:
                    // half c, row r, word j <- column n = 128 c + 32 j + r
                    const long long r0 = (long long)(b * p.blk_stride + p.tok0) * H;
                    const long long nq = (long long)p.rows * H;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t v[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int n = 128 * c + 32 * j + lane;
                            v[j] = (n < N && r0 + n < nq) ? __ldg(p.q_sf + r0 + n) : 0x7f7f7f7fu;
                        }
                        *reinterpret_cast<uint4*>(&sm.sfb[qb][c][lane][0]) =
                            make_uint4(v[0], v[1], v[2], v[3]);
                    }
                    fence_proxy_async_smem();   // read by tcgen05.cp (async proxy)
                }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t bar = smem_u32(&sm.q_full[qb]);
                    mbar_arrive_expect_tx(bar, (uint32_t)(N * elem_bytes(D) + p.tok * H * (p.w_bf16 ? 2 : 4)));
                    // the block's first query row (token b * blk_stride + tok0)
                    const int row0 = b * p.blk_stride + p.tok0;
                    tma_load_2d(smem_u32(sm.q[qb]), &tm_q, bar, 0, row0 * H);
                    tma_load_2d(smem_u32(sm.w[qb]), &tm_w, bar, 0, row0);
                }
                q_blk[k_block & 1] = k_block;
            }
            const int stage = u % S;
            uint32_t ksf[4];
            if (mine) {
                if constexpr (MX && !PAGED) {
                    // the tile's key scales, loaded before the wait for the stage
                    // (the wait hides their latency): word j <- key 32 j + lane
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int key = t * kBlockKV + 32 * j + lane;
                        ksf[j] = key < p.S_kv ? __ldg(p.kv_sf + key) : 0x7f7f7f7fu;
                    }
                }
                // paged: the physical blocks of tile t's pages (-1: none)
                const long long keys = PAGED ? min((long long)ctx, p.width) : 0;
                int ids[4];
                uint32_t bytes = 0;
                auto page_ids = [&]() {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        ids[k] = -1;
                        if (k < ppt) {
                            const int pg = t * ppt + k;
                            if (pg < wbase || pg >= wbase + 32) {   // not sequential: reload
                                wbase = pg & ~31;
                                win0 = page_id(wbase + lane);
                                win1 = page_id(wbase + 32 + lane);
                            }
                            const int id = __shfl_sync(0xffffffffu, win0, pg - wbase);
                            if ((long long)pg * p.block_kv < keys && pg < p.max_blocks) {
                                ids[k] = id;
                                bytes += (uint32_t)(p.block_kv * (elem_bytes(D) + 4));
                            }
                        }
                    }
                };
                if constexpr (PAGED && MX)
                    page_ids();   // the block-table lookups overlap the wait
                if (!warp_wait(smem_u32(&sm.empty[stage]), ((u / S) & 1) ^ 1, wctx, kProducerSleepNs))
                    break;
                const bool last = (u + 1 == n_units) || (t + 1 >= thi);
                const UnitInfo info{b, t, k_block & 1,
                                    (first ? kFirstOfBlock : 0) | (last ? kLastOfBlock : 0)};
                if (PAGED) {
                    // gather the pages of tile t through the block table
                    if constexpr (!MX)
                        page_ids();
                    if (lane == 0) {
                        sm.info[stage] = info;
                        const uint32_t bar = smem_u32(&sm.full[stage]);
                        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (k < ppt && ids[k] >= 0) {
                                tma_load_2d(smem_u32(sm.kv[stage]) + k * p.block_kv * D, &tm_kv, bar, 0,
                                            ids[k] * p.kv_page_rows);
                                // the slots' fp32 scales, or (MX) their scale words:
                                // row ids[k] of the [num_blocks, block_kv] scale map
                                tma_load_2d(smem_u32(&sm.scale[stage][k * p.block_kv]), &tm_scale, bar,
                                            0, ids[k]);
                            }
                        }
                    }
                    // slide the window: the prefetched half becomes current
                    if ((t + 1) * ppt >= wbase + 32) {
                        wbase += 32;
                        win0 = win1;
                        win1 = page_id(wbase + 32 + lane);
                    }
                } else if constexpr (MX) {
                    *reinterpret_cast<uint4*>(&sm.sfa[stage][lane][0]) =
                        make_uint4(ksf[0], ksf[1], ksf[2], ksf[3]);
                    fence_proxy_async_smem();   // read by tcgen05.cp (async proxy)
                    __syncwarp();
                    if (lane == 0) {
                        sm.info[stage] = info;
                        const uint32_t bar = smem_u32(&sm.full[stage]);
                        mbar_arrive_expect_tx(bar, (uint32_t)(kBlockKV * elem_bytes(D)));
                        tma_load_2d(smem_u32(sm.kv[stage]), &tm_kv, bar, 0, t * kBlockKV);
                    }
                } else {
                    if (lane == 0) {
                        sm.info[stage] = info;
                        const uint32_t bar = smem_u32(&sm.full[stage]);
                        mbar_arrive_expect_tx(bar, (uint32_t)(kBlockKV * D + kBlockKV * 4));
                        tma_load_2d(smem_u32(sm.kv[stage]), &tm_kv, bar, 0, t * kBlockKV);
                        tma_load_2d(smem_u32(sm.scale[stage]), &tm_scale, bar, t * kBlockKV, 0);
                    }
                }
            } else if (PAGED) {
                // another producer's unit: keep the page window moving
                if ((t + 1) * ppt >= wbase + 32) {
                    wbase += 32;
                    win0 = win1;
                    win1 = page_id(wbase + 32 + lane);
                }
            }
            u_end = u + 1;
            // advance to the next unit, skipping blocks with no work
            first = false;
            ++t;
            if (t >= thi && u + 1 < n_units) {
                do {
                    ++b;
                    t = 0;
                    enter_block();
                    t = tlo;
                } while (thi <= tlo && b + 1 < p.num_q_blocks);
                if (thi <= tlo)   // ran off the end: the slice disagrees with the inputs
                    break;
                ++k_block;
                first = true;
            }
        }
        // Drain: every copy this warp issued must have landed before exit,
        // also when some role gave up (wait_drain ignores the abort flag).
        if (lane == 0) {
            for (int u = max(0, u_end - S); u < u_end; ++u)
                if (u % kProducers == pid)
                    wait_drain(smem_u32(&sm.full[u % S]), (u / S) & 1, wctx);
            // Only the last two query blocks can still be landing: an older
            // block's buffer was reloaded after its consumers released it,
            // which they did after its copy landed.  (With two producers a
            // buffer's barrier may have moved past an older block's phase, so
            // waiting on that phase would never end.)
            for (int i = 0; i < 2; ++i)
                if (q_blk[i] >= 0 && q_blk[i] >= k_block - 1)
                    wait_drain(smem_u32(&sm.q_full[q_blk[i] & 1]), (q_blk[i] >> 1) & 1, wctx);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= MMA issuer
        regs_dec<kRegsCtl>();
        // Paged MX: the whole warp runs the loop, to put each tile's scale
        // words (copied by TMA in key order) into the transposed rows
        // tcgen05.cp reads; otherwise lane 0 alone.
        constexpr bool kWarpMma = PAGED && MX;
        auto wait = [&](uint32_t bar, uint32_t parity, unsigned sleep) -> bool {
            return kWarpMma ? warp_wait(bar, parity, wctx, sleep) : wait_bounded(bar, parity, wctx, sleep);
        };
        if (kWarpMma || lane == 0) {
            const uint32_t idesc = idesc_e4m3_f32(kBlockKV, (uint32_t)N);
            const uint64_t desc_kv0 = smem_desc(smem_u32(sm.kv[0]), D);
            const uint64_t desc_q0 = smem_desc(smem_u32(sm.q[0]), D);
            int k_block = -1;
            for (int u = 0; u < n_units; ++u) {
                const int stage = u % S;
                if (!wait(smem_u32(&sm.full[stage]), (u / S) & 1, kMmaSleepNs))
                    break;
                const UnitInfo info = sm.info[stage];
                if (info.flags & kFirstOfBlock) {
                    ++k_block;
                    if (!wait(smem_u32(&sm.q_full[info.qbuf]), (k_block >> 1) & 1, 0))
                        break;
                }
                const int buf = u & 1;
                if (!wait(smem_u32(&sm.acc_empty[buf]), ((u >> 1) & 1) ^ 1, kMmaSleepNs))
                    break;
                if constexpr (kWarpMma) {
                    // row lane, word j <- the scale word of key 32 j + lane
                    const uint32_t* lin = reinterpret_cast<const uint32_t*>(sm.scale[stage]);
                    *reinterpret_cast<uint4*>(&sm.sfa[stage][lane][0]) =
                        make_uint4(lin[lane], lin[32 + lane], lin[64 + lane], lin[96 + lane]);
                    fence_proxy_async_smem();   // read by tcgen05.cp (async proxy)
                    __syncwarp();
                    if (lane != 0)
                        continue;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kMaxN);
                // descriptors advance by address / 16: one stage, one query
                // buffer, 32 bytes of K per MMA
                const uint64_t da = desc_kv0 + (uint64_t)(stage * (C::kKVTileBytes >> 4));
                const uint64_t db = desc_q0 + (uint64_t)(info.qbuf * (C::kQTileBytes >> 4));
                if constexpr (MX) {
                    // scale factors into TMEM (in issue order before the MMAs
                    // that read them): the key tile's into the slot of this
                    // unit's parity, the query block's at its first unit
                    const uint32_t sfa_t = tmem_base + kMxSfaCol + (uint32_t)((u & 1) * 4);
                    const uint32_t sfb_t = tmem_base + kMxSfbCol + (uint32_t)(info.qbuf * 8);
                    tmem_cp_32x128b_x4(sfa_t, sf_desc(smem_u32(&sm.sfa[stage][0][0])));
                    if (info.flags & kFirstOfBlock) {
                        tmem_cp_32x128b_x4(sfb_t, sf_desc(smem_u32(&sm.sfb[info.qbuf][0][0][0])));
                        tmem_cp_32x128b_x4(sfb_t + 4, sf_desc(smem_u32(&sm.sfb[info.qbuf][1][0][0])));
                    }
#pragma unroll
                    for (int k = 0; k < D / 32; ++k)
                        mma_mxf8f6f4(d_tmem, da + 2 * k, db + 2 * k,
                                     idesc_mx_f32(kBlockKV, (uint32_t)N, (uint32_t)k, p.mx_fmt), sfa_t,
                                     sfb_t, k > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k = 0; k < D / 32; ++k)
                        mma_f8f6f4(d_tmem, da + 2 * k, db + 2 * k, idesc, k > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&sm.empty[stage]));
                mma_commit(smem_u32(&sm.acc_full[buf]));
                if (info.flags & kLastOfBlock)
                    mma_commit(smem_u32(&sm.q_empty[info.qbuf]));
            }
            // every MMA issued above has completed once this barrier flips;
            // waited for even after an abort, before TMEM is freed
            if (lane == 0) {
                mma_commit(smem_u32(&sm.mma_done));
                wait_drain(smem_u32(&sm.mma_done), 0, wctx);
            }
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ================================================= -inf fill
        regs_dec<kRegsCtl>();
        if (!std::is_same<OutT, CandOut>::value && (p.flags & kFlagClean)) {
            // fill warps: 2 and 3 (dense); 3 alone (paged: warp 2 produces)
            constexpr int nfw = PAGED ? 1 : 2;
            const int fw = warp - (kEpiWarp0 - nfw);
            // paged: the rows of this launch's query atom only
            const int nrows = PAGED ? p.B * p.tok : p.rows;
            for (int rr = cta + fw * G; rr < nrows; rr += nfw * G) {
                const int r = PAGED ? (rr / p.tok) * p.next_n + p.tok0 + rr % p.tok : rr;
                // (candidate instances never fill: the host sets no clean flag)
                using FillT = std::conditional_t<std::is_same<OutT, CandOut>::value, float, OutT>;
                FillT* row = static_cast<FillT*>(p.logits) + (long long)r * p.ldo;
                if (PAGED) {
                    const int c = max(__ldg(p.context_lens + r / p.next_n), 0);
                    const long long covered = min((long long)paged_tiles(c) * kBlockKV, p.width);
                    warp_fill_neg_inf(row, covered, p.width, lane);
                } else if (p.flags & kFlagCompressed) {
                    const int2 rg = dense_range(p, r);
                    warp_fill_neg_inf(row, (long long)(rg.y - rg.x), p.ldo, lane);
                } else {
                    int tlo, thi;
                    int2 mine;
                    dense_block_tiles_warp(p, r / p.tok, lane, tlo, thi, mine);
                    if (thi <= tlo) {
                        warp_fill_neg_inf(row, 0, p.S_kv, lane);
                    } else {
                        warp_fill_neg_inf(row, 0, (long long)tlo * kBlockKV, lane);
                        warp_fill_neg_inf(row, min((long long)thi * kBlockKV, (long long)p.S_kv),
                                          p.S_kv, lane);
                    }
                }
            }
        }
    } else {
        // ================================================= epilogue
        regs_inc<kRegsEpi>();
        // Any negative key scale?  Without one (the usual case: scales are
        // quantisation factors) the epilogue runs the ReLU-by-FMNMX form only
        // and skips the per-unit sign vote.  The paged pool is not scanned; MX
        // calls have no fp32 scale.  The dense scan is the epilogue warps'
        // (all 16 of them: dense units are 256 columns wide), so it overlaps
        // the producer's first copies; their answer meets in shared memory.
        int any_neg = PAGED ? 1 : neg_first;
        if constexpr (!PAGED && !MX && !kScanFirst) {
            const int et = tid - 32 * kEpiWarp0;
            const int n4 = p.S_kv >> 2;
            const float4* s4 = reinterpret_cast<const float4*>(p.kv_scale);
            int neg = 0;
            for (int k = et; k < n4; k += 32 * kNumEpiWarps) {
                const float4 v = __ldg(s4 + k);
                neg |= (v.x < 0.f) | (v.y < 0.f) | (v.z < 0.f) | (v.w < 0.f);
            }
            for (int k = (n4 << 2) + et; k < p.S_kv; k += 32 * kNumEpiWarps)
                neg |= __ldg(p.kv_scale + k) < 0.f;
            if (__any_sync(0xffffffffu, neg) && lane == 0)
                atomicOr(&sm.any_neg, 1);
            __syncwarp();
            mbar_arrive_one_per_warp(smem_u32(&sm.neg_bar));
            any_neg = warp_wait_fast(smem_u32(&sm.neg_bar), 0, wctx)
                          ? *reinterpret_cast<volatile int*>(&sm.any_neg)
                          : 1;   // timed out: the abort flag ends the run anyway
        }
        // Warp group g owns accumulator columns [kEpiCols g, kEpiCols (g + 1)):
        // tokens [g kEpiCols / H, (g + 1) kEpiCols / H) of the unit's query block.
        const int g = (warp - kEpiWarp0) >> 2;
        const int quad = warp & 3;                      // TMEM lanes 32 quad .. 32 quad + 31
        const int tpg = kEpiCols / H;                   // tokens per group
        const int tok0 = g * tpg;
        const int ntok = max(0, min(tpg, p.tok - tok0));
        Epilogue<H, D, MX, OutT> epi{sm, p, wctx,
                           tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(g * kEpiCols),
                           n_units, quad * 32 + lane, g * kEpiCols, tok0, ntok, warp - kEpiWarp0};
        const int nc = ntok * H;   // columns holding tokens, rounded up below
        if (nc > 32) {
            if (any_neg)
                epi.template run<kEpiCols, true>();
            else
                epi.template run<kEpiCols, false>();
        } else if (nc > 16) {
            epi.template run<32, true>();
        } else if (nc > 0) {
            epi.template run<16, true>();
        }   // else: no columns in any unit of this launch; not counted by the barriers
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace mqa
