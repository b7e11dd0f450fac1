// mqa_paged_bf16.cu -- paged instances of the MQA logits kernel with bf16
// logits (each fp32 logit rounded to the nearest even bf16).
#include "launch.h"

namespace mqa {

cudaError_t launch_paged_bf16(int H, int D, const LaunchArgs& a)
{
    if (D == 128) {
        switch (H) {
        case 16: return launch_instance<16, 128, true, false, __nv_bfloat16>(a);
        case 32: return launch_instance<32, 128, true, false, __nv_bfloat16>(a);
        case 64: return launch_instance<64, 128, true, false, __nv_bfloat16>(a);
        }
    } else if (D == 64) {
        switch (H) {
        case 16: return launch_instance<16, 64, true, false, __nv_bfloat16>(a);
        case 32: return launch_instance<32, 64, true, false, __nv_bfloat16>(a);
        case 64: return launch_instance<64, 64, true, false, __nv_bfloat16>(a);
        }
    }
    return cudaErrorNotSupported;
}

}  // namespace mqa
