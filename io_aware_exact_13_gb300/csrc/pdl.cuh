// pdl.cuh -- programmatic dependent launch: a kernel launched with
// launch_dependent() may be scheduled before the kernel ahead of it on the
// stream has finished; it must call grid_dependency_wait() before it touches
// anything that kernel writes. The kernel ahead calls grid_launch_dependents()
// to allow that early scheduling (without it, its completion does).
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace fa {

// This CTA no longer holds back the dependent grid (once every CTA of the grid
// has said so or exited, the dependent grid may be scheduled).
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// Wait until every grid this one depends on has completed and its memory
// operations are visible. Returns at once for a grid launched without the
// dependency.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch kern<<<grid, block, smem, stream>>>(args...) as a programmatic
// dependent of the previous work on the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace fa
