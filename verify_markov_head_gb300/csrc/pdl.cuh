// Programmatic dependent launch: a kernel launched this way may be scheduled
// while the previous kernel on its stream drains, and waits for that
// kernel's completion (and the visibility of its writes) before touching
// global memory.
#pragma once
#include <cuda_runtime.h>
#include <utility>

namespace dspark {

// Blocks until the grids this one depends on programmatically have completed
// and their memory operations are visible; returns at once for a kernel
// launched the ordinary way.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the launch that depends programmatically on this grid start once every
// CTA of this grid has issued it (or exited), instead of at the grid's end.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Launches kern<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialisation.  The kernel must call grid_dependency_wait() before its
// first global-memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace dspark
