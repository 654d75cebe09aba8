// fp32 (TF32 tensor-core) instantiations of the forward kernel. d = 64 only:
// two 128-row fp32 query tiles of d = 128 plus a K/V ring exceed shared memory.
#include "fa_launch.cuh"

namespace fa {
int launch_fwd_fp32(const LaunchArgs &a) {
    if (a.d == 64) return launch_d<float, 64>(a);
    return -4;
}
}  // namespace fa
