/*
 * mqa.h -- C ABI of libmqa.so: FP8 MQA logits scoring (the "lightning indexer"
 * step) on GB300 (sm_103a).
 *
 * The operation ("How to Implement MQA (Multi-Query Attention) Logits
 * Computation with DeepGEMM", instagit article, section "Core Architecture
 * Components": TMA staging, UMMA on E4M3 Q and KV, per-token KV scales, a math
 * reduction that applies ReLU, multiplies by the per-head weight and sums over
 * heads; section "Compressed Logits"):
 *
 *   for query token i and key j with k_start[i] <= j < k_end[i]
 *     logits[i, j] = sum_{h<H} weights[i,h] * ReLU(kv_scale[j] * <q[i,h,:], kv[j,:]>)
 *
 * Positions outside a row's range hold -inf in clean mode ("[PR #435] Improve
 * SM100 MX MQA logits clean-output performance", section "Standalone
 * performance reproducer", which asserts isneginf outside the valid mask and
 * exact zeros inside it for all-zero inputs).
 *
 * Conventions for every call:
 *  - All pointers are DEVICE pointers owned by the caller; the library keeps no
 *    reference after the call returns and allocates no device memory.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously, except under MQA_CHECK_BOUNDS (below).
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns MQA_ERR_INVALID_ARG / MQA_ERR_UNSUPPORTED and
 *    launches nothing.  mqa_last_error_message() explains the last failure of
 *    the calling thread.
 *  - Without MQA_CHECK_BOUNDS, data-dependent inputs are clamped, never trusted:
 *    ranges are intersected with [0, S_kv) (start >= end is an empty row),
 *    context lengths with the block table's capacity, and a block id outside
 *    [0, num_blocks) reads zeros.  No input can make a kernel read or write out
 *    of bounds.
 *  - Kernels never spin without bound: a pipeline wait that runs past its
 *    budget (see mqa_set_wait_limit) stops the kernel and records
 *    MQA_ERR_TIMEOUT, which mqa_device_status() reports.
 */
#ifndef MQA_H
#define MQA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MQA_API __attribute__((visibility("default")))
#else
#define MQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *mqa_stream_t;

typedef enum {
    MQA_OK = 0,
    MQA_ERR_INVALID_ARG = 1, /* bad pointer, size, stride or alignment */
    MQA_ERR_UNSUPPORTED = 2, /* valid request this library has no kernel for */
    MQA_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed */
    MQA_ERR_TIMEOUT = 4,     /* a kernel wait ran out (reported by mqa_device_status) */
    MQA_ERR_BAD_INPUT = 5    /* MQA_CHECK_BOUNDS found an out-of-range input value */
} mqa_status;

enum {
    /* Write -inf to every position of a row that is outside its range (clean
     * logits).  Without it, such positions are left untouched. */
    MQA_CLEAN = 1u,
    /* Dense only: row i stores key k_start[i] + c at column c, c < k_end[i] -
     * k_start[i]; columns [length, ldo) are padding (-inf when MQA_CLEAN). */
    MQA_COMPRESSED = 2u,
    /* Validate data-dependent inputs on the device first (ranges, context
     * lengths, block ids, schedule).  The call then synchronizes `stream` and
     * returns MQA_ERR_BAD_INPUT without computing if any check fails.  Not for
     * use inside CUDA graph capture. */
    MQA_CHECK_BOUNDS = 4u,
    /* Logits as bf16 (each fp32 logit rounded to the nearest even bf16; -inf
     * stays -inf): the `logits` buffer holds 2-byte elements, ldo counts
     * elements.  For mqa_logits, mqa_logits_scheduled, mqa_logits_mx and the
     * paged calls ("[PR #435] ...", section "Validation": FP32/BF16 output).
     * The top-k calls read fp32 logits only. */
    MQA_OUT_BF16 = 16u,
    /* Weights as bf16 ([rows, H] 2-byte elements, 16-byte aligned): each is
     * widened exactly to fp32 and the logits are computed as with fp32
     * weights of the same values.  For mqa_logits, mqa_logits_scheduled,
     * mqa_logits_mx and the paged calls ("[PR #435] ...", section
     * "Validation": FP32/BF16 weights). */
    MQA_WEIGHTS_BF16 = 32u,
    /* Paged FP8 calls: each page of kv_cache holds its block_kv key rows (D
     * E4M3 bytes each) followed by their block_kv fp32 scales, block_kv * (D
     * + 4) bytes in all; kv_scales must be NULL. */
    MQA_KV_FUSED = 64u
};

/*
 * Dense MQA logits ("Implementing Standard MQA Logits Computation" of the
 * instagit article; argument order (q, kv, scales, weights, starts, ends) as in
 * the PR #435 reproducer's call).
 *
 *   q         [S_q, H, D]  FP8 E4M3 bytes, row-major, 16-byte aligned
 *   kv        [S_kv, D]    FP8 E4M3 bytes (one KV head), 16-byte aligned
 *   kv_scale  [S_kv]       fp32 per-key scale, 16-byte aligned
 *   weights   [S_q, H]     fp32 per-(token, head) weight (bf16 with
 *                          MQA_WEIGHTS_BF16), 16-byte aligned
 *   k_start, k_end [S_q]   int32 half-open key range of each query row
 *   logits    [S_q, ldo]   fp32 output, 4-byte aligned (bf16, 2-byte aligned,
 *             with MQA_OUT_BF16).  Uncompressed: row i
 *             has S_kv columns and ldo >= S_kv (columns [S_kv, ldo) are never
 *             written).  Compressed: ldo >= every row's range length.
 *   H in {8, 32, 64}, D in {64, 128}; S_q, S_kv >= 0; S_q * H < 2^31.
 *   flags     MQA_CLEAN | MQA_COMPRESSED | MQA_CHECK_BOUNDS | MQA_OUT_BF16 |
 *             MQA_WEIGHTS_BF16
 */
MQA_API mqa_status mqa_logits(const void *q, const void *kv, const float *kv_scale, const void *weights,
                      const int32_t *k_start, const int32_t *k_end, void *logits, int S_q,
                      int S_kv, int H, int D, int64_t ldo, unsigned flags, mqa_stream_t stream);

/*
 * Dense MQA logits with MX inputs: MXFP8 (E4M3 elements) or, with the flag
 * MQA_MXFP4, MXFP4 (E2M1 elements) ("[PR #435] Improve SM100 MX MQA logits
 * clean-output performance": sections "Performance" (MXFP8 and MXFP4 timings
 * at H=64, D=128) and "Standalone performance reproducer" (q [S_q, H, D] with
 * q_sf [S_q, H] int32, k [S_kv, D] with ks [S_kv] int32, 0x7f7f7f7f = unit
 * scales; MXFP4 elements packed two per byte, D / 2 bytes per row)).
 *
 *   logits[i, j] = sum_h w[i,h] * ReLU(x),  x = sum_b 2^(eq_b - 127) * 2^(ek_b - 127)
 *                                              * sum_{d in block b} q[i,h,d] * kv[j,d]
 *
 *   q        [S_q, H, 128] E4M3 bytes, 16-byte aligned; MXFP4: [S_q, H, 64]
 *            bytes, two E2M1 codes per byte, 32-byte aligned
 *   q_sf     [S_q, H] uint32: byte b (b = 0..3, little end first) is the UE8M0
 *            scale eq_b of elements [32 b, 32 b + 32) of q[i,h,:]; 4-byte aligned
 *   kv       [S_kv, 128] E4M3 bytes, 16-byte aligned; MXFP4: [S_kv, 64] bytes,
 *            32-byte aligned
 *   kv_sf    [S_kv] uint32, the same for kv[j,:]; 16-byte aligned
 *   weights, k_start, k_end, logits, ldo: as mqa_logits.
 *   D is the element count and must be 128; H in {8, 32, 64}.  A scale byte of
 *   255 (not a number in UE8M0) is not allowed.  Which nibble of a byte holds
 *   the lower-indexed element does not change any logit: a 32-element block
 *   is 16 whole bytes, and q and kv pair the same positions.
 *   flags    MQA_CLEAN | MQA_COMPRESSED | MQA_CHECK_BOUNDS | MQA_OUT_BF16 |
 *            MQA_WEIGHTS_BF16 | MQA_MXFP4
 */
enum { MQA_MXFP4 = 8u };   /* flag of mqa_logits_mx: E2M1 elements */
MQA_API mqa_status mqa_logits_mx(const void *q, const uint32_t *q_sf, const void *kv,
                                 const uint32_t *kv_sf, const void *weights,
                                 const int32_t *k_start, const int32_t *k_end, void *logits,
                                 int S_q, int S_kv, int H, int D, int64_t ldo, unsigned flags,
                                 mqa_stream_t stream);

/*
 * Work schedule for a dense call ("[PR #435] Improve SM100 MX MQA logits
 * clean-output performance": the reproducer computes get_mqa_logits_metadata
 * once outside the timed region and passes it to the logits call as
 * schedule_meta; section "Validation" checks that the scheduled path gives the
 * same output as the unscheduled one).  The pages fix neither its layout nor
 * its unit; this library's:
 *
 * A query block b is the tok = 256 / H query rows [b * tok, (b + 1) * tok)
 * (the last one may be short); it spans the 128-key tiles from the first to
 * the last key of any of its rows (ranges intersected with [0, S_kv), start >=
 * end empty).  A unit is one block against one tile of its span, numbered
 * block by block, U in total.  SM k starts at unit floor(k * U / num_sms);
 * entry k is that unit's (block, absolute tile index); entry num_sms, and any
 * entry at U, is (number of blocks, 0).
 *
 *   k_start, k_end [S_q] int32 (device): the ranges the logits call will get
 *   schedule_meta  [num_sms + 1][2] int32 (device), written by this call
 *   H in {8, 32, 64}; num_sms >= 1 (normally mqa_get_num_sms()).
 */
MQA_API mqa_status mqa_logits_metadata(const int32_t *k_start, const int32_t *k_end, int S_q,
                                       int S_kv, int H, int num_sms, int32_t *schedule_meta,
                                       mqa_stream_t stream);

/*
 * mqa_logits with a precomputed schedule: CTA k of the num_sms launched
 * processes the units between entries k and k + 1 of schedule_meta (from
 * mqa_logits_metadata for the same k_start, k_end, S_q, S_kv, H and num_sms)
 * instead of deriving its slice from all the ranges.  Every output element is
 * computed with the same arithmetic either way: the results are bitwise
 * identical to mqa_logits.  The kernel checks that the entries it reads are
 * ordered and inside the blocks' spans (an inconsistent schedule records
 * MQA_ERR_BAD_INPUT for mqa_device_status and computes nothing); under
 * MQA_CHECK_BOUNDS the whole schedule is recomputed and compared first.
 * Other arguments and errors: as mqa_logits.
 */
MQA_API mqa_status mqa_logits_scheduled(const void *q, const void *kv, const float *kv_scale,
                                        const void *weights, const int32_t *k_start,
                                        const int32_t *k_end, const int32_t *schedule_meta,
                                        int num_sms, void *logits, int S_q, int S_kv, int H,
                                        int D, int64_t ldo, unsigned flags, mqa_stream_t stream);

/*
 * Work schedule for paged_mqa_logits ("[PR #314] fix: SM90 paged MQA logits
 * IMA on next_n=4", sections "a97b74d" Root cause / Fix: schedule_meta holds
 * num_sms + 1 entries and host and kernel must agree on the query atom).
 *
 * A work unit is one sequence's next_n query tokens against one 128-key tile;
 * sequence b owns ceil(max(context_lens[b], 0) / 128) units, numbered sequence
 * by sequence.  SM k starts at unit floor(k * U / num_sms) of U in total and
 * entry k is that unit's (sequence, tile) pair; entry num_sms, and any entry at
 * U, is (B, 0).  next_n and block_kv only select validation here.
 *
 *   context_lens  [B] int32 (device)
 *   schedule_meta [num_sms + 1][2] int32 (device), written by this call
 *   block_kv in {32, 64, 128}; num_sms >= 1 (normally mqa_get_num_sms()).
 */
MQA_API mqa_status paged_mqa_logits_metadata(const int32_t *context_lens, int B, int next_n, int block_kv,
                                     int num_sms, int32_t *schedule_meta, mqa_stream_t stream);

/*
 * Paged decode MQA logits ("Implementing Paged MQA Logits Computation for
 * Decoding" of the instagit article; next_n queries per sequence and block_kv
 * pages as in "[PR #314] ...", section "12cb7c0").
 *
 *   q            [B * next_n, H, D] FP8 E4M3 bytes, 16-byte aligned; row
 *                r = b * next_n + t is query t of sequence b
 *   kv_cache     [num_blocks, block_kv, D] FP8 E4M3 bytes, 16-byte aligned
 *   kv_scales    [num_blocks, block_kv] fp32, 16-byte aligned
 *                (with MQA_KV_FUSED: kv_cache is [num_blocks, block_kv * (D +
 *                4)] bytes, a page's key rows then their scales, and
 *                kv_scales is NULL; the same logits as the separate layout)
 *   weights      [B * next_n, H] fp32 (bf16 with MQA_WEIGHTS_BF16), 16-byte
 *                aligned
 *   context_lens [B] int32
 *   block_table  [B, max_blocks_per_seq] int32: logical page p of sequence b
 *                lives in physical block block_table[b, p]
 *   schedule_meta the output of paged_mqa_logits_metadata for the same
 *                context_lens, next_n, block_kv and num_sms
 *   logits       [B * next_n, ldo] fp32; a row has max_blocks_per_seq *
 *                block_kv columns, ldo >= that.  Row r scores key positions
 *                [0, context_lens[b] - next_n + t + 1); key position j is slot
 *                j % block_kv of block block_table[b, j / block_kv].
 *   H in {16, 32, 64}, D in {64, 128}, 1 <= next_n <= 64, block_kv in
 *   {32, 64, 128}.  A sequence's next_n tokens are scored in query atoms of
 *   at most 256 / H tokens (one kernel launch per atom over the same
 *   schedule), as "[PR #314] ...", section "a97b74d", splits next_n into
 *   query atoms.
 *   num_sms      the number of schedule_meta entries minus one (the schedule's
 *                length; the kernel runs one CTA per entry).  Not in the pages'
 *                call, where the schedule tensor carries its own shape.
 *   flags        MQA_CLEAN | MQA_CHECK_BOUNDS | MQA_OUT_BF16 | MQA_WEIGHTS_BF16
 *                | MQA_KV_FUSED (MQA_COMPRESSED is rejected)
 */
MQA_API mqa_status paged_mqa_logits(const void *q, const void *kv_cache, const float *kv_scales,
                            const void *weights, const int32_t *context_lens,
                            const int32_t *block_table, int max_blocks_per_seq,
                            const int32_t *schedule_meta, void *logits, int B, int next_n, int H,
                            int D, int block_kv, int num_blocks, int num_sms, int64_t ldo,
                            unsigned flags, mqa_stream_t stream);

/*
 * Paged decode MQA logits with MX keys and queries: MXFP8 (E4M3) or, with the
 * flag MQA_MXFP4, MXFP4 (E2M1, two codes per byte) elements and UE8M0 block
 * scales ("[PR #314] fix: SM90 paged MQA logits IMA on next_n=4", section
 * "Testing": the paged logits are tested with FP4 keys on GB200; the element
 * and scale encoding as mqa_logits_mx).  Row r = b * next_n + t scores key
 * positions [0, context_lens[b] - next_n + t + 1) with
 *   x = sum_b 2^(eq_b - 127) * 2^(ek_b - 127) * sum_{d in block b} q[r,h,d] * kv[j,d]
 * in place of kv_scale * <q, kv>; everything else as paged_mqa_logits.
 *
 *   q         [B * next_n, H, 128] E4M3 bytes (16-byte aligned), or with
 *             MQA_MXFP4 [B * next_n, H, 64] packed E2M1 bytes (32-byte aligned)
 *   q_sf      [B * next_n, H] uint32, four UE8M0 scales each; 4-byte aligned
 *   kv_cache  [num_blocks, block_kv, 128] E4M3 bytes, or [.., 64] packed E2M1
 *             (alignment as q)
 *   kv_sf     [num_blocks, block_kv] uint32: the scale word of each key slot,
 *             beside its key as kv_scales is for FP8 keys; 16-byte aligned
 *   D must be 128; H in {16, 32, 64}; query atoms of at most 192 / H tokens
 *   (the scale factors share the accumulator memory).
 *   flags     MQA_CLEAN | MQA_CHECK_BOUNDS | MQA_OUT_BF16 | MQA_WEIGHTS_BF16 |
 *             MQA_MXFP4
 */
MQA_API mqa_status paged_mqa_logits_mx(const void *q, const uint32_t *q_sf, const void *kv_cache,
                                       const uint32_t *kv_sf, const void *weights,
                                       const int32_t *context_lens, const int32_t *block_table,
                                       int max_blocks_per_seq, const int32_t *schedule_meta,
                                       void *logits, int B, int next_n, int H, int D, int block_kv,
                                       int num_blocks, int num_sms, int64_t ldo, unsigned flags,
                                       mqa_stream_t stream);

/*
 * Paged decode MQA logits without any caller-provided or library-allocated
 * scratch (the pages have no counterpart to this call; it is an addition of
 * this library).  Arguments are those of paged_mqa_logits minus
 * schedule_meta and num_sms: the work schedule is written into a fixed array
 * in the library's own device memory (a file-scope static device array of
 * MQA_NOALLOC_MAX_SMS + 1 entries that every GPU loading the library holds
 * until the process exits) and the paged kernel reads it from there.
 *
 * For callers that cannot allocate device memory: a C host program or plugin
 * that has no handle to the framework's allocator owning the GPU, a decode loop
 * that must not call cudaMalloc because it may implicitly synchronize the
 * device in the middle of a step, or a service with a fixed, pre-planned
 * device-memory budget.  The call itself allocates nothing and calls no
 * allocating routine.
 *
 * - The first call on a device looks up the array's device address (with that
 *   device current); make that first call before any stream capture.
 * - Devices with more than MQA_NOALLOC_MAX_SMS SMs are rejected with
 *   MQA_ERR_UNSUPPORTED.
 * - Every call on a device shares the one array: calls whose work overlaps on
 *   the GPU (different streams without ordering) race on it.  Each call
 *   rewrites every entry it uses, so no state from an earlier call leaks in.
 */
#define MQA_NOALLOC_MAX_SMS 1024
MQA_API mqa_status paged_mqa_logits_noalloc(const void *q, const void *kv_cache,
                                            const float *kv_scales, const void *weights,
                                            const int32_t *context_lens,
                                            const int32_t *block_table, int max_blocks_per_seq,
                                            void *logits, int B, int next_n, int H, int D,
                                            int block_kv, int num_blocks, int64_t ldo,
                                            unsigned flags, mqa_stream_t stream);

/*
 * Top-k keys per query row of dense MQA logits: the `indices` that the
 * sparse-attention call on the "FlashMLA" page consumes (parameters of
 * flash_mla_with_kvcache: shape (batch, seq_len_q, topk), invalid entries set
 * to -1).  The pages fix only that contract; this library reads it as:
 *
 *   row i of `indices` holds the min(topk, len_i) keys j of the row's range
 *   with the largest logits[i, j], in ascending key order, then -1 up to topk.
 *   "Largest" follows the IEEE-754 totalOrder of the fp32 value (-NaN < -inf
 *   < ... < -0 < +0 < ... < +inf < +NaN); among equal values the smaller key
 *   is taken, so the result is unique.
 *
 *   logits   [S_q, ldo] fp32, 4-byte aligned: the output of mqa_logits
 *   k_start, k_end [S_q] int32: the ranges given to mqa_logits, intersected
 *            with [0, S_kv) in the same way (start >= end: no keys)
 *   indices  [S_q, topk] int32 output, 4-byte aligned
 *   S_kv     keys of an uncompressed row, ldo >= S_kv.  With MQA_COMPRESSED
 *            key j of row i is read at column j - k_start[i], and a range
 *            longer than ldo is cut at k_start[i] + ldo.
 *   topk >= 1; flags: MQA_COMPRESSED (MQA_CLEAN is accepted and has no
 *   effect; MQA_CHECK_BOUNDS is rejected).
 * The logits are only read; positions outside the ranges are never read.
 */
MQA_API mqa_status mqa_topk_indices(const float *logits, const int32_t *k_start,
                                    const int32_t *k_end, int32_t *indices, int S_q, int S_kv,
                                    int64_t ldo, int topk, unsigned flags, mqa_stream_t stream);

/*
 * Top-k keys per row of paged decode logits (the output of paged_mqa_logits):
 * row r = b * next_n + t selects among keys [0, context_lens[b] - next_n + t +
 * 1) intersected with [0, width), with the rules of mqa_topk_indices.
 *
 *   logits       [B * next_n, ldo] fp32, 4-byte aligned; width <= ldo keys a row
 *   context_lens [B] int32
 *   indices      [B * next_n, topk] int32 output, 4-byte aligned
 */
MQA_API mqa_status paged_mqa_topk_indices(const float *logits, const int32_t *context_lens,
                                          int32_t *indices, int B, int next_n, int width,
                                          int64_t ldo, int topk, mqa_stream_t stream);

/*
 * Fused logits + top-k over dense KV: the `indices` of mqa_topk_indices for
 * the logits mqa_logits would compute (non-clean, uncompressed), without
 * writing those logits.  The top-k follows the MQA logits directly in the
 * indexer: "FlashMLA", parameters of flash_mla_with_kvcache (indices of shape
 * (batch, seq_len_q, topk), -1 for invalid entries), over the logits of "How
 * to Implement MQA (Multi-Query Attention) Logits Computation with DeepGEMM",
 * section "Core Architecture Components".
 *
 *   q, kv, kv_scale, weights, k_start, k_end, S_q, S_kv, H, D: as mqa_logits
 *            (ranges are clamped to [0, S_kv] as mqa_topk_indices clamps them)
 *   indices  [S_q, topk] int32 output, 4-byte aligned
 *   topk >= 1
 *   workspace  device memory of at least mqa_logits_topk_workspace_size(S_q,
 *            S_kv) bytes, 256-byte aligned, owned by the caller; its contents
 *            on entry do not matter and on return are unspecified.  It holds
 *            one fp32 slot per key of every row (rows padded to a multiple of
 *            128 keys), a 32-bit mask per 32 keys and a few words per row, but
 *            only the candidates are written: for each row the logits of a
 *            tail of its range (max(2 topk, sqrt(len topk)) keys, at a 128-key
 *            boundary) and those of the rest not below the topk-th largest
 *            logit of that tail.
 *   flags: MQA_WEIGHTS_BF16 or 0 (others are rejected).
 * The result equals mqa_topk_indices applied to the mqa_logits output for the
 * same inputs, bit for bit (both compute each logit with the same
 * arithmetic).  Five kernels on `stream`; no host synchronisation.  Errors:
 * invalid sizes, pointers, alignment or flags return MQA_ERR_INVALID_ARG and
 * unsupported H or D MQA_ERR_UNSUPPORTED before anything is launched; a
 * kernel wait that runs out is reported by mqa_device_status.
 */
MQA_API size_t mqa_logits_topk_workspace_size(int S_q, int S_kv);
MQA_API mqa_status mqa_logits_topk(const void *q, const void *kv, const float *kv_scale,
                                   const void *weights, const int32_t *k_start,
                                   const int32_t *k_end, int32_t *indices, void *workspace,
                                   size_t workspace_bytes, int S_q, int S_kv, int H, int D,
                                   int topk, unsigned flags, mqa_stream_t stream);

/* Number of SMs of `device` (cached), or -1 on error. */
MQA_API int mqa_get_num_sms(int device);

/* Synchronizes `stream`, then returns and clears the current device's kernel
 * status word: MQA_ERR_TIMEOUT if a kernel wait ran out, MQA_ERR_BAD_INPUT if
 * a bounds check failed, MQA_OK otherwise. */
MQA_API mqa_status mqa_device_status(mqa_stream_t stream);

/* Budget, in SM clock cycles, of every pipeline wait in kernels launched after
 * this call (default 4e9, about two seconds).  0 restores the default. */
MQA_API mqa_status mqa_set_wait_limit(unsigned long long cycles);

/* Test hook for the timeout path: launches one CTA that waits, with the given
 * budget, on a barrier nothing ever signals.  The wait runs out, the kernel
 * exits cleanly and the next mqa_device_status() returns MQA_ERR_TIMEOUT. */
MQA_API mqa_status mqa_selftest_wait_timeout(unsigned long long cycles, mqa_stream_t stream);

MQA_API const char *mqa_status_string(mqa_status s);

/* Human-readable reason for the last non-OK status returned to this thread. */
MQA_API const char *mqa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* MQA_H */
