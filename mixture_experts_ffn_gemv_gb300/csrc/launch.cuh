// Kernel launches with programmatic dependent launch (PDL): each kernel is
// launched with programmatic stream serialization, so the next kernel on the
// stream is scheduled while this one drains.  Every kernel calls pdl_wait()
// before it reads anything an earlier kernel wrote (it returns once those
// grids have completed and their writes are visible) and pdl_trigger() to let
// its own successor be scheduled.  Without PDL both are no-ops.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
