// cluster.cuh -- thread-block cluster barrier helpers and the cluster launch
// used by the kernels whose CTAs share one Q/K head (decode.cu, sequential.cu).
#pragma once

#include <cuda_runtime.h>

namespace gdn {

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 256-thread CTAs in clusters of csize along x (no cluster attribute when csize == 1).
// With dependent set, the kernel is a programmatic dependent of the previous kernel in
// the stream: it may start once that kernel's CTAs have all signalled (or ended), and
// waits (griddepcontrol.wait) before it reads anything that kernel may write (only
// constant layer parameters are read before the wait).
template <typename K, typename A>
static cudaError_t launch_cluster(K kernel, dim3 grid, int csize, cudaStream_t s, const A &args,
                                  bool dependent = false)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (csize > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = csize;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (dependent) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

// The two halves of a programmatic dependency, in a kernel launched as above.
__device__ __forceinline__ void wait_previous_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" :::); }

}  // namespace gdn
