// launch.h -- host-side launch interface between the C ABI (mqa_api.cu) and the
// kernel instantiations (mqa_dense.cu, mqa_paged.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "mqa_kernel.cuh"

namespace mqa {

struct LaunchArgs {
    CUtensorMap tm_q;
    CUtensorMap tm_kv;
    CUtensorMap tm_scale;
    CUtensorMap tm_w;
    Params p;
    int grid;
    cudaStream_t stream;
};

// Both return cudaErrorNotSupported for an (H, D) pair without an instance.
cudaError_t launch_dense(int H, int D, const LaunchArgs& a);
cudaError_t launch_paged(int H, int D, const LaunchArgs& a);

template <int H, int D, bool PAGED>
cudaError_t launch_instance(const LaunchArgs& a)
{
    auto kern = mqa_logits_kernel<H, D, PAGED>;
    const size_t smem = sizeof(Smem<D>) + 1024;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_kv, a.tm_scale, a.tm_w, a.p);
    return cudaGetLastError();
}

}  // namespace mqa
