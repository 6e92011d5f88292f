// launch.cuh -- kernel launch with the library's launch attributes.
//
// Every GEMM/GEMV kernel is launched with programmatic stream serialisation
// (unless SDT_PDL=0): the kernel's set-up (barrier initialisation, TMEM
// allocation, descriptor prefetch) may then overlap the tail of the previous
// kernel in the stream, and the kernel executes griddepcontrol.wait before its
// first global-memory access, so it still observes all of that kernel's
// results.  Cluster dimensions are added for two-CTA tiles.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <utility>

namespace sdt {

inline bool pdl_enabled() {
    static const bool on = [] {
        const char *s = getenv("SDT_PDL");
        return !(s && (!strcmp(s, "0") || !strcmp(s, "off")));
    }();
    return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sdt
