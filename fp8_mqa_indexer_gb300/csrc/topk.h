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

}  // namespace mqa
