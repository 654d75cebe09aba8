// fp16 instantiations of the forward with an additive mask: the 128-key-block
// kernel on the mask's packed one-bit form, and the 64-key-block kernel on the
// fp32 mask (a mask with values other than 0 and -inf, or a per-head bias).
#include "fa_launch.cuh"

namespace fa {
int launch_fwd_mask_fp16(const LaunchArgs &a) {
    if (a.d == 128) return launch_mask_fwd_d<__half, 128>(a);
    if (a.d == 64) return launch_mask_fwd_d<__half, 64>(a);
    return -4;
}
}  // namespace fa
