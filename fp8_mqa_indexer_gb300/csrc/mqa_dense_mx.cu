// mqa_dense_mx.cu -- MXFP8 (block-scaled E4M3) dense instances of the MQA
// logits kernel.
#include "launch.h"

namespace mqa {

cudaError_t launch_dense_mx(int H, bool bf16, const LaunchArgs& a)
{
    if (bf16) {
        switch (H) {
        case 8: return launch_instance<8, 128, false, true, __nv_bfloat16>(a);
        case 32: return launch_instance<32, 128, false, true, __nv_bfloat16>(a);
        case 64: return launch_instance<64, 128, false, true, __nv_bfloat16>(a);
        }
        return cudaErrorNotSupported;
    }
    switch (H) {
    case 8: return launch_instance<8, 128, false, true>(a);
    case 32: return launch_instance<32, 128, false, true>(a);
    case 64: return launch_instance<64, 128, false, true>(a);
    }
    return cudaErrorNotSupported;
}

}  // namespace mqa
