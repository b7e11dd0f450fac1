/*
 * mqa_oracle.c -- plain, slow CPU oracle for MQA logits scoring.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no header, constant or helper with the CUDA library.
 *
 * What it computes (sources are the four web pages this project is built from):
 *
 *   "How to Implement MQA (Multi-Query Attention) Logits Computation with
 *    DeepGEMM" (instagit), section "Core Architecture Components":
 *      - the score of query token i against KV token j is the per-head dot
 *        product of q[i,h,:] with the single KV head kv[j,:], passed through a
 *        ReLU, multiplied by the per-head weight w[i,h] and summed over heads
 *        ("Math Warp Reduction");
 *      - per-token fp32 KV scales are applied to the dot product (FAQ "How does
 *        DeepGEMM handle quantization scales");
 *      - compressed logits keep only [k_start, k_end) of each row
 *        ("Compressed Logits").
 *   "[PR #435] Improve SM100 MX MQA logits clean-output performance", section
 *   "Standalone performance reproducer": positions outside a row's range are
 *   -inf in clean mode, and all-zero inputs give exactly 0 inside the range.
 *
 * Written out, for k_start[i] <= j < k_end[i]:
 *
 *     logits[i, j] = sum_h  w[i,h] * max(0, s[j] * sum_d q[i,h,d] * kv[j,d])
 *
 * with q and kv decoded exactly from FP8 E4M3 (torch.float8_e4m3fn), and every
 * step in double precision.  The inner dot product is exact in double: each
 * product of two E4M3 values is a multiple of 2^-18 below 2^18, so any partial
 * sum of up to 2^16 terms is an integer multiple of 2^-18 below 2^34, which a
 * 53-bit significand holds exactly (D above 2^16 is rejected).  The head sum
 * is rounded once to fp32 at the end.
 *
 * Readings this oracle takes where the pages are silent or disagree:
 *   - fill value outside the range is -inf (the reproducer's isneginf assert),
 *     not the zero-fill one sentence of the instagit article mentions;
 *   - the scale sits inside the ReLU, exactly as in the formula above;
 *   - a range is intersected with [0, S_kv); start >= end is an empty row;
 *   - the paged decode row t of sequence b scores keys [0, ctx_b - next_n + t + 1);
 *   - in non-clean mode positions outside the range are left untouched.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>

#define ORACLE_CLEAN 1u
#define ORACLE_COMPRESSED 2u

/* ---------------------------------------------------------------------------
 * FP8 E4M3 ("fn" variant, as torch.float8_e4m3fn): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits, no infinities, codes 0x7F / 0xFF are NaN.
 *   exponent field 0      : subnormal, value = mantissa * 2^-9
 *   exponent field 1..15  : normal,    value = (8 + mantissa) * 2^(exp - 10)
 * The largest finite value is (8 + 6) * 2^5 = 448.
 * ------------------------------------------------------------------------- */
static double e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant, -9);
    else
        mag = ldexp((double)(8 + mant), expo - 10);
    return sign ? -mag : mag;
}

/* The 256 decoded values, built once from e4m3_decode (a lookup, not a
 * different decoding). */
static double g_table[256];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;

static void build_table(void)
{
    for (int c = 0; c < 256; ++c)
        g_table[c] = e4m3_decode((uint8_t)c);
}

static const double *table(void)
{
    pthread_once(&g_table_once, build_table);
    return g_table;
}

int oracle_e4m3_table(double *out256)
{
    const double *t = table();
    for (int c = 0; c < 256; ++c)
        out256[c] = t[c];
    return 0;
}

static void decode_row(const uint8_t *src, size_t n, double *dst)
{
    const double *t = table();
    for (size_t k = 0; k < n; ++k)
        dst[k] = t[src[k]];
}

/* Exact dot product of two decoded E4M3 vectors of length D (see header
 * comment), summed in order d = 0 .. D-1. */
static double dot(const double *a, const double *b, int D)
{
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
        acc += a[d] * b[d];
    return acc;
}

/* One logit and its tolerance term sum_h |w * s * x|; q_dec is the decoded
 * [H, D] query row, kv_dec the decoded key. */
static float one_logit(const double *q_dec, const double *kv_dec, double s, const float *w_row,
                       int H, int D, double *abs_sum)
{
    double sum = 0.0, asum = 0.0;
    for (int h = 0; h < H; ++h) {
        double x = dot(q_dec + (size_t)h * D, kv_dec, D);
        double sx = s * x;
        double r = sx > 0.0 ? sx : 0.0;
        sum += (double)w_row[h] * r;
        asum += fabs((double)w_row[h] * sx);
    }
    if (abs_sum)
        *abs_sum = asum;
    return (float)sum;
}

/*
 * Dense MQA logits for rows [row_begin, row_end).
 *   q        [S_q, H, D] E4M3 bytes      kv       [S_kv, D] E4M3 bytes
 *   kv_scale [S_kv] fp32                 weights  [S_q, H] fp32
 *   k_start, k_end [S_q] int32
 *   logits   points at row row_begin of an [.., ldo] fp32 matrix
 *   tol      (nullable) same layout as logits, receives 1e-3*sum_h|w s x| + 1e-5
 *            at every written logit position
 * Uncompressed: row i has S_kv columns (ldo >= S_kv).  Compressed: column c of
 * row i holds key k_start[i] + c; clean mode fills c in [len_i, ldo) with -inf.
 * Returns 0, or -1 on invalid arguments.
 */
int oracle_mqa_logits(const uint8_t *q, const uint8_t *kv, const float *kv_scale,
                      const float *weights, const int32_t *k_start, const int32_t *k_end,
                      int S_q, int S_kv, int H, int D, int64_t ldo, unsigned flags,
                      int row_begin, int row_end, float *logits, double *tol)
{
    int clean = (flags & ORACLE_CLEAN) != 0;
    int compressed = (flags & ORACLE_COMPRESSED) != 0;
    if (S_q < 0 || S_kv < 0 || H <= 0 || D <= 0 || D > 65536 || row_begin < 0 || row_end > S_q ||
        row_begin > row_end)
        return -1;
    if (!compressed && ldo < S_kv)
        return -1;
    if (compressed && ldo < 0)
        return -1;
    double *q_dec = malloc(sizeof(double) * (size_t)H * D);
    double *kv_dec = malloc(sizeof(double) * (size_t)D);
    if (!q_dec || !kv_dec) {
        free(q_dec);
        free(kv_dec);
        return -2;
    }
    int rc = 0;
    for (int i = row_begin; i < row_end && rc == 0; ++i) {
        float *out = logits + (size_t)(i - row_begin) * (size_t)ldo;
        double *tout = tol ? tol + (size_t)(i - row_begin) * (size_t)ldo : NULL;
        int lo = k_start[i] < 0 ? 0 : k_start[i];
        int hi = k_end[i] > S_kv ? S_kv : k_end[i];
        if (hi < lo)
            hi = lo;
        if (compressed && (int64_t)(hi - lo) > ldo) {
            rc = -1;
            break;
        }
        decode_row(q + (size_t)i * H * D, (size_t)H * D, q_dec);
        int64_t width = compressed ? ldo : S_kv;
        for (int64_t c = 0; c < width; ++c) {
            int j = compressed ? (int)(lo + c) : (int)c;
            int valid = compressed ? (c < hi - lo) : (j >= lo && j < hi);
            if (valid) {
                double asum;
                decode_row(kv + (size_t)j * D, (size_t)D, kv_dec);
                out[c] = one_logit(q_dec, kv_dec, (double)kv_scale[j], weights + (size_t)i * H, H, D,
                                   &asum);
                if (tout)
                    tout[c] = 1e-3 * asum + 1e-5;
            } else if (clean) {
                out[c] = -INFINITY;
                if (tout)
                    tout[c] = 0.0;
            }
        }
    }
    free(q_dec);
    free(kv_dec);
    return rc;
}

/*
 * Paged decode MQA logits ("Implementing Paged MQA Logits Computation for
 * Decoding" of the instagit article; next_n and block_kv as in "[PR #314] fix:
 * SM90 paged MQA logits IMA on next_n=4").  Rows are r = b * next_n + t.
 *   q          [B * next_n, H, D] E4M3      weights [B * next_n, H] fp32
 *   kv_cache   [num_blocks, block_kv, D] E4M3
 *   kv_scales  [num_blocks, block_kv] fp32
 *   context_lens [B] int32
 *   block_table  [B, max_blocks_per_seq] int32: logical page -> physical block
 * Row r scores key positions j in [0, context_lens[b] - next_n + t + 1); key j
 * lives in block block_table[b, j / block_kv], slot j % block_kv.  A row has
 * max_blocks_per_seq * block_kv columns; clean mode writes -inf elsewhere.
 * Returns 0, or -1 on invalid arguments (including a block id out of range or a
 * context longer than the block table).
 */
int oracle_paged_mqa_logits(const uint8_t *q, const uint8_t *kv_cache, const float *kv_scales,
                            const float *weights, const int32_t *context_lens,
                            const int32_t *block_table, int max_blocks_per_seq, int B, int next_n,
                            int H, int D, int block_kv, int num_blocks, int64_t ldo,
                            unsigned flags, int row_begin, int row_end, float *logits, double *tol)
{
    int clean = (flags & ORACLE_CLEAN) != 0;
    int64_t width = (int64_t)max_blocks_per_seq * block_kv;
    if (B < 0 || next_n <= 0 || H <= 0 || D <= 0 || D > 65536 || block_kv <= 0 || num_blocks < 0 ||
        max_blocks_per_seq < 0 || ldo < width || row_begin < 0 || row_end > B * next_n ||
        row_begin > row_end || (flags & ORACLE_COMPRESSED))
        return -1;
    double *q_dec = malloc(sizeof(double) * (size_t)H * D);
    double *kv_dec = malloc(sizeof(double) * (size_t)D);
    if (!q_dec || !kv_dec) {
        free(q_dec);
        free(kv_dec);
        return -2;
    }
    int rc = 0;
    for (int r = row_begin; r < row_end && rc == 0; ++r) {
        int b = r / next_n, t = r % next_n;
        int ctx = context_lens[b];
        if (ctx < 0 || (int64_t)ctx > width) {
            rc = -1;
            break;
        }
        decode_row(q + (size_t)r * H * D, (size_t)H * D, q_dec);
        int end = ctx - next_n + t + 1;
        if (end < 0)
            end = 0;
        float *out = logits + (size_t)(r - row_begin) * (size_t)ldo;
        double *tout = tol ? tol + (size_t)(r - row_begin) * (size_t)ldo : NULL;
        for (int64_t j = 0; j < width; ++j) {
            if (j < end) {
                int32_t blk = block_table[(size_t)b * max_blocks_per_seq + j / block_kv];
                if (blk < 0 || blk >= num_blocks) {
                    rc = -1;
                    break;
                }
                size_t tok = (size_t)blk * block_kv + (size_t)(j % block_kv);
                double asum;
                decode_row(kv_cache + tok * D, (size_t)D, kv_dec);
                out[j] = one_logit(q_dec, kv_dec, (double)kv_scales[tok], weights + (size_t)r * H, H, D,
                                   &asum);
                if (tout)
                    tout[j] = 1e-3 * asum + 1e-5;
            } else if (clean) {
                out[j] = -INFINITY;
                if (tout)
                    tout[j] = 0.0;
            }
        }
    }
    free(q_dec);
    free(kv_dec);
    return rc;
}

/*
 * Paged work schedule.  The pages fix its shape -- num_sms + 1 entries, entry k
 * saying where SM k starts and entry num_sms marking the end ("[PR #314] ...",
 * section "a97b74d", "Fix": schedule_meta sized num_sms + 1) -- but not the unit
 * of work.  This library's reading: a unit is one sequence's next_n queries
 * against one 128-key tile, sequence b owns ceil(max(ctx_b, 0) / 128) units,
 * units are numbered sequence by sequence, and SM k starts at unit
 * floor(k * U / num_sms) of U in total.  Entry k is the pair (b, tile) of that
 * unit; the end entry, and any start at U, is (B, 0).
 * next_n and block_kv do not change the split (a whole sequence is one query
 * atom); they are validated only.  Returns 0, or -1 on invalid arguments.
 */
int oracle_paged_mqa_logits_metadata(const int32_t *context_lens, int B, int next_n, int block_kv,
                                     int num_sms, int32_t *schedule_meta /* [num_sms + 1, 2] */)
{
    if (B < 0 || next_n <= 0 || block_kv <= 0 || 128 % block_kv != 0 || num_sms <= 0)
        return -1;
    int64_t total = 0;
    for (int b = 0; b < B; ++b) {
        int ctx = context_lens[b] > 0 ? context_lens[b] : 0;
        total += (ctx + 127) / 128;
    }
    for (int k = 0; k <= num_sms; ++k) {
        int64_t u = (int64_t)k * total / num_sms;
        int64_t before = 0;
        int b = 0;
        int32_t tile = 0;
        for (; b < B; ++b) {
            int ctx = context_lens[b] > 0 ? context_lens[b] : 0;
            int64_t n = (ctx + 127) / 128;
            if (u < before + n) {
                tile = (int32_t)(u - before);
                break;
            }
            before += n;
        }
        schedule_meta[2 * k] = b;            /* b == B when u == total */
        schedule_meta[2 * k + 1] = b < B ? tile : 0;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Dense work schedule, the counterpart of the paged one for mqa_logits ("[PR
 * #435] ...", section "Standalone performance reproducer", which builds
 * get_mqa_logits_metadata(starts, ends, ...) once and passes it as
 * schedule_meta; section "Validation", scheduled-path equality).  The pages fix
 * neither its layout nor its unit; this library's reading, with the same
 * num_sms + 1 shape as the paged schedule:
 *   - a query block is tok = 256 / H consecutive query rows (block b holds rows
 *     [b * tok, min(S_q, (b + 1) * tok)));
 *   - the keys of a row are its range intersected with [0, S_kv) (start >= end:
 *     no keys); block b spans the 128-key tiles from the first key of any of
 *     its rows to the last: tiles [min lo / 128, ceil(max hi / 128)), none if
 *     every row is empty;
 *   - a unit is one block against one tile of its span; units are numbered
 *     block by block, tile by tile, U in total;
 *   - SM k starts at unit floor(k * U / num_sms); entry k is that unit's
 *     (block, tile) with the tile's absolute index; the end entry, and any
 *     start at U, is (num_blocks, 0).
 * Returns 0, or -1 on invalid arguments.
 * ------------------------------------------------------------------------- */
static void dense_block_span(const int32_t *k_start, const int32_t *k_end, int S_q, int S_kv,
                             int tok, int b, int64_t *t_lo, int64_t *t_hi)
{
    int64_t lo_min = -1, hi_max = -1;
    for (int i = b * tok; i < S_q && i < (b + 1) * tok; ++i) {
        int64_t lo = k_start[i] < 0 ? 0 : k_start[i];
        int64_t hi = k_end[i] > S_kv ? S_kv : k_end[i];
        if (lo > S_kv)
            lo = S_kv;
        if (hi <= lo)
            continue;
        if (lo_min < 0 || lo < lo_min)
            lo_min = lo;
        if (hi > hi_max)
            hi_max = hi;
    }
    if (lo_min < 0) {
        *t_lo = *t_hi = 0;
    } else {
        *t_lo = lo_min / 128;
        *t_hi = (hi_max + 127) / 128;
    }
}

int oracle_mqa_logits_metadata(const int32_t *k_start, const int32_t *k_end, int S_q, int S_kv,
                               int H, int num_sms, int32_t *schedule_meta /* [num_sms + 1, 2] */)
{
    if (S_q < 0 || S_kv < 0 || H <= 0 || H > 256 || 256 % H != 0 || num_sms <= 0)
        return -1;
    const int tok = 256 / H;
    const int nb = (S_q + tok - 1) / tok;
    int64_t total = 0;
    for (int b = 0; b < nb; ++b) {
        int64_t lo, hi;
        dense_block_span(k_start, k_end, S_q, S_kv, tok, b, &lo, &hi);
        total += hi - lo;
    }
    for (int k = 0; k <= num_sms; ++k) {
        const int64_t u = (int64_t)k * total / num_sms;
        int64_t before = 0;
        int b = 0;
        int32_t tile = 0;
        for (; b < nb; ++b) {
            int64_t lo, hi;
            dense_block_span(k_start, k_end, S_q, S_kv, tok, b, &lo, &hi);
            if (u < before + (hi - lo)) {
                tile = (int32_t)(lo + (u - before));
                break;
            }
            before += hi - lo;
        }
        schedule_meta[2 * k] = b;            /* b == nb when u == total */
        schedule_meta[2 * k + 1] = b < nb ? tile : 0;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Top-k key selection per query row: the step that consumes the logits.  The
 * "FlashMLA" page (parameters of flash_mla_with_kvcache) fixes only its
 * output contract: `indices` of shape (batch, seq_len_q, topk) naming the keys
 * each query attends to, with invalid entries set to -1.  Readings this
 * oracle takes, since the pages leave the rest open:
 *   - the candidates of row i are the keys of its range [lo, hi), normalised as
 *     for the logits (intersected with [0, n_cols); in the compressed layout key
 *     j sits at column j - lo and the range stops at lo + ldo);
 *   - "top" means the largest logits under the IEEE-754 totalOrder of the fp32
 *     value (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN), and among equal
 *     values (the same bit pattern) the smaller key index comes first;
 *   - the first min(topk, hi - lo) keys of that order are written in
 *     ascending key order, followed by -1 up to topk.
 * ------------------------------------------------------------------------- */

/* Rank of an fp32 bit pattern in totalOrder: non-negative values by their
 * magnitude bits, negative values below every non-negative one and reversed. */
static int64_t total_order_rank(float v)
{
    union {
        float f;
        uint32_t u;
    } b;
    b.f = v;
    int64_t mag = (int64_t)(b.u & 0x7fffffffu);
    return (b.u >> 31) ? -mag - 1 : mag;
}

typedef struct {
    int64_t rank;
    int32_t key;
} ranked_key;

/* Larger rank first; equal ranks by smaller key. */
static int by_rank_then_key(const void *pa, const void *pb)
{
    const ranked_key *a = pa, *b = pb;
    if (a->rank != b->rank)
        return a->rank > b->rank ? -1 : 1;
    return (a->key > b->key) - (a->key < b->key);
}

/*
 * Top-k keys of rows [row_begin, row_end).
 *   logits  [rows, ldo] fp32 (row i starts at logits + i * ldo)
 *   k_start, k_end [rows] int32 key ranges; n_cols = keys per uncompressed row
 *   flags   ORACLE_COMPRESSED: key j of row i is at column j - lo, and the
 *           range is cut at lo + ldo
 *   out     points at row row_begin of an [.., topk] int32 matrix
 * Returns 0, or -1 on invalid arguments.
 */
int oracle_topk_indices(const float *logits, int64_t ldo, const int32_t *k_start,
                        const int32_t *k_end, int rows, int n_cols, unsigned flags, int topk,
                        int row_begin, int row_end, int32_t *out)
{
    int compressed = (flags & ORACLE_COMPRESSED) != 0;
    if (rows < 0 || n_cols < 0 || topk <= 0 || ldo < 0 || row_begin < 0 || row_end > rows ||
        row_begin > row_end || (!compressed && ldo < n_cols))
        return -1;
    ranked_key *cand = malloc(sizeof(ranked_key) * (size_t)(n_cols > 0 ? n_cols : 1));
    unsigned char *chosen = malloc((size_t)(n_cols > 0 ? n_cols : 1));
    if (!cand || !chosen) {
        free(cand);
        free(chosen);
        return -2;
    }
    for (int i = row_begin; i < row_end; ++i) {
        int lo = k_start[i] < 0 ? 0 : (k_start[i] > n_cols ? n_cols : k_start[i]);
        int hi = k_end[i] > n_cols ? n_cols : k_end[i];
        if (hi < lo)
            hi = lo;
        if (compressed && (int64_t)(hi - lo) > ldo)
            hi = (int)(lo + ldo);
        const float *row = logits + (size_t)i * (size_t)ldo;
        int n = hi - lo;
        for (int c = 0; c < n; ++c) {
            int j = lo + c;
            cand[c].rank = total_order_rank(row[compressed ? c : j]);
            cand[c].key = j;
        }
        qsort(cand, (size_t)n, sizeof(ranked_key), by_rank_then_key);
        int take = n < topk ? n : topk;
        for (int c = 0; c < n; ++c)
            chosen[c] = 0;
        for (int c = 0; c < take; ++c)
            chosen[cand[c].key - lo] = 1;
        int32_t *o = out + (size_t)(i - row_begin) * (size_t)topk;
        int pos = 0;
        for (int c = 0; c < n; ++c)
            if (chosen[c])
                o[pos++] = lo + c;
        while (pos < topk)
            o[pos++] = -1;
    }
    free(cand);
    free(chosen);
    return 0;
}

/* ---------------------------------------------------------------------------
 * MX variant of the dense logits ("[PR #435] Improve SM100 MX MQA logits
 * clean-output performance", sections "Performance" and "Standalone
 * performance reproducer"): q and kv carry microscaling block scales instead
 * of a per-key fp32 scale.  The reproducer fixes the shapes: q [S_q, H, D]
 * elements with one int32 per (row, head) holding four UE8M0 scale bytes for
 * D = 128, kv [S_kv, D] with one int32 per key, and 0x7f7f7f7f meaning every
 * scale is one.  Readings this oracle takes where the pages are silent:
 *   - a block is 32 consecutive elements of D, and byte b of the int32 (bits
 *     8b .. 8b+7) scales block b;
 *   - a UE8M0 byte e scales by 2^(e - 127) (e = 255 is not a number);
 *   - MXFP8 elements are E4M3 as above; MXFP4 elements are E2M1 (1 sign, 2
 *     exponent bits with bias 1, 1 mantissa bit), two per byte, element 2c in
 *     the low nibble of byte c;
 *   - the score is the same ReLU, weight and head sum with the block-scaled dot
 *     product in place of s[j] * <q, kv>:
 *       x = sum_b 2^(eq_b - 127) * 2^(ek_b - 127) * sum_{d in block b} q[d] kv[d].
 * Each block's sum is exact (E4M3 or E2M1 products are integers after scaling
 * by 2^18, 32 of them stay below 2^43), the blocks combine in double.
 * ------------------------------------------------------------------------- */

/* E2M1: value = (-1)^s * (m * 0.5) when the exponent field is 0, else
 * (-1)^s * 2^(e - 1) * (1 + m / 2). */
static double e2m1_decode(unsigned code)
{
    int sign = (code >> 3) & 1;
    int expo = (code >> 1) & 3;
    int mant = code & 1;
    double mag = expo == 0 ? 0.5 * mant : ldexp(1.0 + 0.5 * mant, expo - 1);
    return sign ? -mag : mag;
}

int oracle_e2m1_table(double *out16)
{
    for (unsigned c = 0; c < 16; ++c)
        out16[c] = e2m1_decode(c);
    return 0;
}

/* Element d of a row of D elements: E4M3 byte d, or nibble d of the packed
 * E2M1 bytes (low nibble first). */
static double mx_element(const uint8_t *row, int d, int fp4)
{
    if (!fp4)
        return table()[row[d]];
    uint8_t byte = row[d / 2];
    return e2m1_decode((d & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0xF));
}

/* Block-scaled dot product of a query row and a key row (D elements each). */
static double mx_dot(const uint8_t *qrow, uint32_t qsf, const uint8_t *krow, uint32_t ksf, int D,
                     int fp4)
{
    double x = 0.0;
    for (int b = 0; b < D / 32; ++b) {
        int64_t acc = 0; /* block sum, in units of 2^-18 */
        for (int d = 32 * b; d < 32 * b + 32; ++d)
            acc += (int64_t)llround(ldexp(mx_element(qrow, d, fp4), 9)) *
                   (int64_t)llround(ldexp(mx_element(krow, d, fp4), 9));
        int eq = (int)((qsf >> (8 * b)) & 0xFF), ek = (int)((ksf >> (8 * b)) & 0xFF);
        if (eq == 255 || ek == 255)
            return NAN;
        x += ldexp((double)acc, eq + ek - 254 - 18);
    }
    return x;
}

/*
 * MX dense logits for rows [row_begin, row_end); layout and flags as
 * oracle_mqa_logits.
 *   q     [S_q, H, D] E4M3 bytes, or [S_q, H, D/2] packed E2M1 when fp4
 *   q_sf  [S_q, H] uint32, four UE8M0 block scales each
 *   kv    [S_kv, D] E4M3 bytes, or [S_kv, D/2] packed E2M1 when fp4
 *   kv_sf [S_kv] uint32
 * D must be 128 (four blocks).  tol receives 1e-3 * sum_h |w x| + 1e-5.
 */
int oracle_mx_mqa_logits(const uint8_t *q, const uint32_t *q_sf, const uint8_t *kv,
                         const uint32_t *kv_sf, const float *weights, const int32_t *k_start,
                         const int32_t *k_end, int S_q, int S_kv, int H, int D, int fp4,
                         int64_t ldo, unsigned flags, int row_begin, int row_end, float *logits,
                         double *tol)
{
    int clean = (flags & ORACLE_CLEAN) != 0;
    int compressed = (flags & ORACLE_COMPRESSED) != 0;
    if (S_q < 0 || S_kv < 0 || H <= 0 || D != 128 || row_begin < 0 || row_end > S_q ||
        row_begin > row_end || (!compressed && ldo < S_kv) || (compressed && ldo < 0))
        return -1;
    const size_t row_bytes = (size_t)(fp4 ? D / 2 : D);
    for (int i = row_begin; i < row_end; ++i) {
        float *out = logits + (size_t)(i - row_begin) * (size_t)ldo;
        double *tout = tol ? tol + (size_t)(i - row_begin) * (size_t)ldo : NULL;
        int lo = k_start[i] < 0 ? 0 : k_start[i];
        int hi = k_end[i] > S_kv ? S_kv : k_end[i];
        if (hi < lo)
            hi = lo;
        if (compressed && (int64_t)(hi - lo) > ldo)
            return -1;
        int64_t width = compressed ? ldo : S_kv;
        for (int64_t c = 0; c < width; ++c) {
            int j = compressed ? (int)(lo + c) : (int)c;
            int valid = compressed ? (c < hi - lo) : (j >= lo && j < hi);
            if (valid) {
                double sum = 0.0, asum = 0.0;
                for (int h = 0; h < H; ++h) {
                    double x = mx_dot(q + ((size_t)i * H + h) * row_bytes, q_sf[(size_t)i * H + h],
                                      kv + (size_t)j * row_bytes, kv_sf[j], D, fp4);
                    double w = (double)weights[(size_t)i * H + h];
                    sum += w * (x > 0.0 ? x : 0.0);
                    asum += fabs(w * x);
                }
                out[c] = (float)sum;
                if (tout)
                    tout[c] = 1e-3 * asum + 1e-5;
            } else if (clean) {
                out[c] = -INFINITY;
                if (tout)
                    tout[c] = 0.0;
            }
        }
    }
    return 0;
}

/*
 * Paged MX logits for rows [row_begin, row_end): the paged decode of
 * oracle_paged_mqa_logits with the block-scaled scores of oracle_mx_mqa_logits
 * ("[PR #314] fix: SM90 paged MQA logits IMA on next_n=4", section "Testing":
 * the paged MQA logits are tested with FP4 keys on GB200; the element and
 * scale encoding is the one read above for the dense MX call).  Reading taken:
 * the per-key UE8M0 scale word sits beside its key in the paged layout, one
 * uint32 per slot of a block, as the per-key fp32 scale does for FP8 keys.
 *   q         [B * next_n, H, D] E4M3 bytes, or [.., D/2] packed E2M1 when fp4
 *   q_sf      [B * next_n, H] uint32, four UE8M0 block scales each
 *   kv_cache  [num_blocks, block_kv, D] E4M3 bytes, or [.., D/2] packed E2M1
 *   kv_sf     [num_blocks, block_kv] uint32
 * Row r = b * next_n + t scores key positions [0, ctx_b - next_n + t + 1);
 * position j is slot j % block_kv of block block_table[b, j / block_kv].
 * D must be 128.  tol receives 1e-3 * sum_h |w x| + 1e-5.
 */
int oracle_paged_mx_mqa_logits(const uint8_t *q, const uint32_t *q_sf, const uint8_t *kv_cache,
                               const uint32_t *kv_sf, const float *weights,
                               const int32_t *context_lens, const int32_t *block_table,
                               int max_blocks_per_seq, int B, int next_n, int H, int D, int fp4,
                               int block_kv, int num_blocks, int64_t ldo, unsigned flags,
                               int row_begin, int row_end, float *logits, double *tol)
{
    int clean = (flags & ORACLE_CLEAN) != 0;
    int64_t width = (int64_t)max_blocks_per_seq * block_kv;
    if (B < 0 || next_n <= 0 || H <= 0 || D != 128 || block_kv <= 0 || num_blocks < 0 ||
        max_blocks_per_seq < 0 || ldo < width || row_begin < 0 || row_end > B * next_n ||
        row_begin > row_end || (flags & ORACLE_COMPRESSED))
        return -1;
    const size_t row_bytes = (size_t)(fp4 ? D / 2 : D);
    for (int r = row_begin; r < row_end; ++r) {
        int b = r / next_n, t = r % next_n;
        int ctx = context_lens[b];
        if (ctx < 0 || (int64_t)ctx > width)
            return -1;
        int end = ctx - next_n + t + 1;
        if (end < 0)
            end = 0;
        float *out = logits + (size_t)(r - row_begin) * (size_t)ldo;
        double *tout = tol ? tol + (size_t)(r - row_begin) * (size_t)ldo : NULL;
        for (int64_t j = 0; j < width; ++j) {
            if (j < end) {
                int32_t blk = block_table[(size_t)b * max_blocks_per_seq + j / block_kv];
                if (blk < 0 || blk >= num_blocks)
                    return -1;
                size_t slot = (size_t)blk * block_kv + (size_t)(j % block_kv);
                double sum = 0.0, asum = 0.0;
                for (int h = 0; h < H; ++h) {
                    double x = mx_dot(q + ((size_t)r * H + h) * row_bytes, q_sf[(size_t)r * H + h],
                                      kv_cache + slot * row_bytes, kv_sf[slot], D, fp4);
                    double w = (double)weights[(size_t)r * H + h];
                    sum += w * (x > 0.0 ? x : 0.0);
                    asum += fabs(w * x);
                }
                out[j] = (float)sum;
                if (tout)
                    tout[j] = 1e-3 * asum + 1e-5;
            } else if (clean) {
                out[j] = -INFINITY;
                if (tout)
                    tout[j] = 0.0;
            }
        }
    }
    return 0;
}
