// fp16 instantiations of the forward for packed variable-length batches
// (the 128-key-block kernel).
#include "fa_launch.cuh"

namespace fa {
int launch_fwd_varlen_fp16(const LaunchArgs &a) {
    if (a.d == 128) return launch_bk128_d<__half, 128, true>(a);
    if (a.d == 64) return launch_bk128_d<__half, 64, true>(a);
    return -4;
}
}  // namespace fa
