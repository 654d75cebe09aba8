// fp16 instantiations of the forward kernel for packed variable-length batches.
#include "fa_launch.cuh"

namespace fa {
int launch_fwd_varlen_fp16(const LaunchArgs &a) {
    if (a.d == 128) return launch_varlen_d<__half, 128>(a);
    if (a.d == 64) return launch_varlen_d<__half, 64>(a);
    return -4;
}
}  // namespace fa
