// mqa_dense.cu -- dense-KV instances of the MQA logits kernel.
#include "launch.h"

namespace mqa {

cudaError_t launch_dense(int H, int D, bool bf16, const LaunchArgs& a)
{
    if (bf16)
        return launch_dense_bf16(H, D, a);
    if (D == 128) {
        switch (H) {
        case 8: return launch_instance<8, 128, false>(a);
        case 32: return launch_instance<32, 128, false>(a);
        case 64: return launch_instance<64, 128, false>(a);
        }
    } else if (D == 64) {
        switch (H) {
        case 8: return launch_instance<8, 64, false>(a);
        case 32: return launch_instance<32, 64, false>(a);
        case 64: return launch_instance<64, 64, false>(a);
        }
    }
    return cudaErrorNotSupported;
}

}  // namespace mqa
