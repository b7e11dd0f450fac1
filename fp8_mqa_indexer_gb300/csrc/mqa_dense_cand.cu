// mqa_dense_cand.cu -- dense instances of the MQA logits kernel that write
// candidates for the fused logits + top-k call: per 32-key line, the logits at
// or above the row's threshold packed to the front of the line and a mask of
// their keys.
#include "launch.h"

namespace mqa {

cudaError_t launch_dense_cand(int H, int D, const LaunchArgs& a)
{
    if (D == 128) {
        switch (H) {
        case 8: return launch_instance<8, 128, false, false, CandOut>(a);
        case 32: return launch_instance<32, 128, false, false, CandOut>(a);
        case 64: return launch_instance<64, 128, false, false, CandOut>(a);
        }
    } else if (D == 64) {
        switch (H) {
        case 8: return launch_instance<8, 64, false, false, CandOut>(a);
        case 32: return launch_instance<32, 64, false, false, CandOut>(a);
        case 64: return launch_instance<64, 64, false, false, CandOut>(a);
        }
    }
    return cudaErrorNotSupported;
}

}  // namespace mqa
