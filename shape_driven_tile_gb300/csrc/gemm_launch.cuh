// gemm_launch.cuh -- body of the per-tile host launcher; each gemm_t*.cu
// instantiates it for one tile so the ladder compiles in parallel.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "gemm_kernel.cuh"

namespace sdt {

template <int BM, int BN>
int launch_gemm_tile(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &args,
                     cudaStream_t stream) {
    using Cfg = TileCfg<BM, BN>;
    auto kern = gemm_f16_tile_kernel<BM, BN>;
    const int smem = Cfg::smem_bytes(args.stages);
    // Raise the dynamic shared-memory cap once per device to the largest this launch needs.
    static std::atomic<int> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (configured[dev].load(std::memory_order_acquire) < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int prev = configured[dev].load();
        while (prev < smem && !configured[dev].compare_exchange_weak(prev, smem)) {
        }
    }
    const unsigned grid = static_cast<unsigned>(args.num_m_tiles) * static_cast<unsigned>(args.num_n_tiles);
    kern<<<grid, Cfg::THREADS, smem, stream>>>(tmA, tmB, args);
    return cudaGetLastError();
}

}  // namespace sdt

#define SDT_INSTANTIATE_GEMM_TILE(BM, BN)                                                          \
    template int sdt::launch_gemm_tile<BM, BN>(const CUtensorMap &, const CUtensorMap &,           \
                                               const sdt::GemmArgs &, cudaStream_t);
