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
template <typename K, typename A>
static cudaError_t launch_cluster(K kernel, dim3 grid, int csize, cudaStream_t s, const A &args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = csize > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

}  // namespace gdn
