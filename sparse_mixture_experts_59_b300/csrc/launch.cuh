// launch.cuh -- kernel launches with programmatic dependent launch (and
// optionally a cluster shape), the host side of pdl_wait / pdl_trigger.
#pragma once

#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <utility>

namespace moe {

// PDL is on unless the environment sets MOE_PDL=0.
inline bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("MOE_PDL");
        return !(e && strcmp(e, "0") == 0);
    }();
    return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, int cluster_x, Args&&... args) {
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
