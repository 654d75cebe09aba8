// bf16 instantiations of the forward: the 128-key-block kernel without a mask,
// the 64-key-block kernel with an additive mask.
#include "fa_launch.cuh"

namespace fa {
int launch_fwd_bf16(const LaunchArgs &a) {
    if (a.mask) {
        if (a.d == 128) return launch_masked_d<__nv_bfloat16, 128>(a);
        if (a.d == 64) return launch_masked_d<__nv_bfloat16, 64>(a);
        return -4;
    }
    if (a.d == 128) return launch_bk128_d<__nv_bfloat16, 128, false>(a);
    if (a.d == 64) return launch_bk128_d<__nv_bfloat16, 64, false>(a);
    return -4;
}
}  // namespace fa
