// mqa_paged_mx.cu -- paged-KV (decode) instances of the MQA logits kernel with
// MX (block-scaled E4M3 or E2M1) keys and queries.
#include "launch.h"

namespace mqa {

cudaError_t launch_paged_mx(int H, bool bf16, const LaunchArgs& a)
{
    if (bf16) {
        switch (H) {
        case 16: return launch_instance<16, 128, true, true, __nv_bfloat16>(a);
        case 32: return launch_instance<32, 128, true, true, __nv_bfloat16>(a);
        case 64: return launch_instance<64, 128, true, true, __nv_bfloat16>(a);
        }
        return cudaErrorNotSupported;
    }
    switch (H) {
    case 16: return launch_instance<16, 128, true, true>(a);
    case 32: return launch_instance<32, 128, true, true>(a);
    case 64: return launch_instance<64, 128, true, true>(a);
    }
    return cudaErrorNotSupported;
}

}  // namespace mqa
