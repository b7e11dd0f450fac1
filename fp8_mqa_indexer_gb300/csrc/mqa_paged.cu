// mqa_paged.cu -- paged-KV (decode) instances of the MQA logits kernel.
#include "launch.h"

namespace mqa {

cudaError_t launch_paged(int H, int D, bool bf16, const LaunchArgs& a)
{
    if (bf16)
        return launch_paged_bf16(H, D, a);
    if (D == 128) {
        switch (H) {
        case 16: return launch_instance<16, 128, true>(a);
        case 32: return launch_instance<32, 128, true>(a);
        case 64: return launch_instance<64, 128, true>(a);
        }
    } else if (D == 64) {
        switch (H) {
        case 16: return launch_instance<16, 64, true>(a);
        case 32: return launch_instance<32, 64, true>(a);
        case 64: return launch_instance<64, 64, true>(a);
        }
    }
    return cudaErrorNotSupported;
}

}  // namespace mqa
