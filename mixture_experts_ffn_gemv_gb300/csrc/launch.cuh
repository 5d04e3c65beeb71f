// Kernel launches with programmatic dependent launch (PDL): each kernel is
// launched with programmatic stream serialization, so the next kernel on the
// stream is scheduled while this one drains.  Every kernel calls pdl_wait()
// before it reads anything an earlier kernel wrote (it returns once those
// grids have completed and their writes are visible) and pdl_trigger() to let
// its own successor be scheduled.  Without PDL both are no-ops.
#pragma once

#include <cuda_runtime.h>

#include <mutex>
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

// Whether all `blocks` blocks of `kernel` can be resident at once (one wave).
// Only such a kernel triggers its successor before its own wait: its
// successor's blocks, parked in their waits, then cannot take the slots that
// later blocks of this kernel would need.  Occupancy per (kernel, block size,
// shared memory) is computed once.
inline bool one_wave(const void* kernel, int blocks, int threads, size_t smem) {
    struct Entry {
        const void* k;
        int threads;
        size_t smem;
        int slots;
    };
    static Entry cache[32];
    static int n = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].k == kernel && cache[i].threads == threads && cache[i].smem == smem)
            return blocks <= cache[i].slots;
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const int slots = per_sm * sms;
    if (n < 32) cache[n++] = Entry{kernel, threads, smem, slots};
    return blocks <= slots;
}

}  // namespace moe
