// launch.h -- host-side launch interface between the C ABI (mqa_api.cu) and the
// kernel instantiations (mqa_dense.cu, mqa_paged.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

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
// bf16: __nv_bfloat16 logits instead of float.
cudaError_t launch_dense(int H, int D, bool bf16, const LaunchArgs& a);
cudaError_t launch_paged(int H, int D, bool bf16, const LaunchArgs& a);
cudaError_t launch_paged_mx(int H, bool bf16, const LaunchArgs& a);
cudaError_t launch_dense_mx(int H, bool bf16, const LaunchArgs& a);
cudaError_t launch_dense_bf16(int H, int D, const LaunchArgs& a);
cudaError_t launch_paged_bf16(int H, int D, const LaunchArgs& a);
// candidate instances (CandOut) of the fused logits + top-k call
cudaError_t launch_dense_cand(int H, int D, const LaunchArgs& a);

template <int H, int D, bool PAGED, bool MX = false, typename OutT = float>
cudaError_t launch_instance(const LaunchArgs& a)
{
    auto kern = mqa_logits_kernel<H, D, PAGED, MX, OutT>;
    const size_t smem = sizeof(Smem<D, MX>) + 1024;
    // The shared-memory limit is a per-device attribute of the function: set it
    // once on each device (one bit per device; setting it twice is harmless).
    static std::atomic<unsigned long long> attr_set{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (!(attr_set.load() & bit) || !bit) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set.fetch_or(bit);
    }
    {
        // a programmatic dependent of the preceding kernel in the stream (the
        // work schedule, for paged and scheduled dense calls): see
        // grid_dependency_wait in the kernel
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = a.stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_kv, a.tm_scale, a.tm_w, a.p);
    }
}

}  // namespace mqa
