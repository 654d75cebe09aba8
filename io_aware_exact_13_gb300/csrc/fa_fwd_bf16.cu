// bf16 instantiations of the forward without a mask (the 128-key-block kernel);
// a forward with a mask goes to fa_fwd_mask_bf16.cu.
#include "fa_launch.cuh"

namespace fa {
int launch_fwd_bf16(const LaunchArgs &a) {
    if (a.mask) return launch_fwd_mask_bf16(a);
    if (a.d == 128) return launch_bk128_d<__nv_bfloat16, 128, false>(a);
    if (a.d == 64) return launch_bk128_d<__nv_bfloat16, 64, false>(a);
    return -4;
}
}  // namespace fa
