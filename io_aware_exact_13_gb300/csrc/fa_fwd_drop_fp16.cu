// fp16 instantiations of the forward with dropout (the 128-key-block kernel).
#include "fa_launch.cuh"

namespace fa {
int launch_fwd_drop_fp16(const LaunchArgs &a) {
    if (a.d == 128) return launch_drop_fwd_d<__half, 128>(a);
    if (a.d == 64) return launch_drop_fwd_d<__half, 64>(a);
    return -4;
}
}  // namespace fa
