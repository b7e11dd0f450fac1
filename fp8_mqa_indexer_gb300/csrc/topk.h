// topk.h -- host-side interface of the top-k key selection kernel (mqa_topk.cu).
#pragma once
#include <cuda_runtime.h>

namespace mqa {

struct TopkParams {
    const float* logits;      // [rows, ldo] fp32
    long long ldo;
    int rows;
    int n_cols;               // keys of an uncompressed row
    const int* k_start;       // dense: [rows] key ranges (nullptr when paged)
    const int* k_end;
    const int* context_lens;  // paged: [rows / next_n] (nullptr when dense)
    int next_n;
    int compressed;           // key j of row i sits at column j - k_start[i]
    int topk;
    int* indices;             // [rows, topk] int32 output
};

constexpr int kTopkThreads = 256;
constexpr int kTopkCtasPerSm = 4;

cudaError_t launch_topk(const TopkParams& p, int grid, cudaStream_t stream);

// The fused logits + top-k call (mqa_logits_topk).  Row i's range [lo, hi)
// (k_start / k_end clamped to [0, n_cols]) is split at a 128-key boundary s
// into a prefix [s, hi) of at least max(2 topk, sqrt(n topk)) keys and a
// remainder [lo, s).  The plain logits kernel writes every logit of the
// prefix at its own column; the threshold kernel sets thr[i] to the order key
// of the prefix's topk-th largest logit (thr_f[i]: that logit); the candidate
// logits kernel then writes the remainder's logits not below thr_f[i], packed
// at the front of each 32-key line, with a mask of their keys; the select
// kernel takes the topk
// largest of the prefix's logits and the remainder's candidates.  Rows with at
// most topk keys have empty prefix and remainder.
struct CandTopkParams {
    const int* k_start;       // [rows] the call's key ranges
    const int* k_end;
    int rows;
    int n_cols;               // keys (S_kv)
    int topk;
    long long ldo;            // candidate row stride in floats, a multiple of 128
    float* vals;              // [rows, ldo] prefix logits at their own columns; remainder
                              // line L packs its kept logits at 32 L
    unsigned* mask;           // [rows + 1, ldo / 32] keys kept in each remainder line
    int* pre_lo;              // [rows] prefix ranges
    int* pre_hi;
    int* rem_lo;              // [rows] remainder ranges
    int* rem_hi;
    unsigned* thr;            // [rows] threshold keys
    float* thr_f;             // [rows] the same thresholds as fp32 values
    unsigned* t0;             // [rows] selection hint: a key about 1.4 topk keys clear (0: none)
    int* indices;             // [rows, topk] int32 output
};

cudaError_t launch_cand_split(const CandTopkParams& p, cudaStream_t stream);
cudaError_t launch_cand_threshold(const CandTopkParams& p, int grid, cudaStream_t stream);
cudaError_t launch_cand_select(const CandTopkParams& p, int grid, cudaStream_t stream);

}  // namespace mqa
