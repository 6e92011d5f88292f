// gemm_launch.cuh -- body of the per-tile host launcher; each gemm_t*.cu
// instantiates it for one tile so the ladder compiles in parallel.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "gemm_kernel.cuh"
#include "gemm_persistent.cuh"
#include "gemm_pair.cuh"
#include "gemm_streamk.cuh"
#include "launch.cuh"

namespace sdt {

// Raise a kernel's dynamic shared-memory cap once per device (and kernel) to the
// largest size a launch has asked for.
template <typename Kern>
int ensure_smem(Kern kern, int smem, std::atomic<int> *configured) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (configured[dev].load(std::memory_order_acquire) < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int prev = configured[dev].load();
        while (prev < smem && !configured[dev].compare_exchange_weak(prev, smem)) {
        }
    }
    return cudaSuccess;
}

template <int BM, int BN, int LAYOUT>
int launch_gemm_tile(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &, const GemmArgs &args,
                     cudaStream_t stream) {
    using Cfg = TileCfg<BM, BN>;
    auto kern = gemm_f16_tile_kernel<BM, BN, false, LAYOUT>;
    const int smem = Cfg::smem_bytes(args.stages);
    static std::atomic<int> configured[64];
    if (int e = ensure_smem(kern, smem, configured)) return e;
    const unsigned grid = static_cast<unsigned>(args.num_m_tiles) * static_cast<unsigned>(args.num_n_tiles);
    return launch_kernel(kern, dim3(grid), dim3(Cfg::THREADS), size_t(smem), stream, 1, tmA, tmB, args);
}

// Split-K form.
template <int BM, int BN, int LAYOUT>
int launch_gemm_tile_split(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &args,
                           cudaStream_t stream) {
    using Cfg = TileCfg<BM, BN>;
    auto kern = gemm_f16_tile_kernel<BM, BN, true, LAYOUT>;
    const int smem = Cfg::smem_bytes(args.stages);
    static std::atomic<int> configured[64];
    if (int e = ensure_smem(kern, smem, configured)) return e;
    const dim3 grid(static_cast<unsigned>(args.num_m_tiles) * static_cast<unsigned>(args.num_n_tiles),
                    static_cast<unsigned>(args.splits), 1);
    return launch_kernel(kern, grid, dim3(Cfg::THREADS), size_t(smem), stream, 1, tmA, tmB, args);
}

// Stream-K form: args.splits CTAs share the (tile, k-tile) units.
template <int BM, int BN, int LAYOUT>
int launch_gemm_streamk(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &args,
                        cudaStream_t stream) {
    using Cfg = StreamCfg<BM, BN>;
    auto kern = gemm_streamk_kernel<BM, BN, LAYOUT>;
    const int smem = Cfg::smem_bytes(args.stages);
    static std::atomic<int> configured[64];
    if (int e = ensure_smem(kern, smem, configured)) return e;
    return launch_kernel(kern, dim3(static_cast<unsigned>(args.splits)), dim3(Cfg::THREADS), size_t(smem), stream, 1,
                         tmA, tmB, args);
}

template <int BN, int LAYOUT>
int launch_gemm_persistent(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                           const GemmArgs &args, cudaStream_t stream) {
    using Cfg = PersistentCfg<BN>;
    auto kern = gemm_f16_persistent_kernel<BN, LAYOUT>;
    const int smem = Cfg::smem_bytes(args.stages);
    static std::atomic<int> configured[64];
    if (int e = ensure_smem(kern, smem, configured)) return e;
    const long long tiles = static_cast<long long>(args.num_m_tiles) * args.num_n_tiles;
    const unsigned grid = static_cast<unsigned>(tiles < args.max_ctas ? tiles : args.max_ctas);
    return launch_kernel(kern, dim3(grid), dim3(Cfg::THREADS), size_t(smem), stream, 1, tmA, tmB, tmC, args);
}

template <int BN, int LAYOUT>
int launch_gemm_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &args,
                     cudaStream_t stream) {
    using Cfg = PairCfg<BN>;
    // the form with the k-split last round only when the plan splits it
    const bool ksplit = args.tail_splits >= 2;
    auto kern = ksplit ? gemm_f16_pair_kernel<BN, LAYOUT, true> : gemm_f16_pair_kernel<BN, LAYOUT, false>;
    const int smem = Cfg::smem_bytes(args.stages);
    static std::atomic<int> configured[2][64];
    if (int e = ensure_smem(kern, smem, configured[ksplit ? 1 : 0])) return e;
    const long long items = args.num_items;
    const long long pairs_cap = args.max_ctas / 2 > 0 ? args.max_ctas / 2 : 1;
    const unsigned pairs = static_cast<unsigned>(items < pairs_cap ? items : pairs_cap);
    return launch_kernel(kern, dim3(2 * pairs), dim3(Cfg::THREADS), size_t(smem), stream, 2, tmA, tmB, tmC, args);
}

}  // namespace sdt

// Each macro instantiates one ladder tile for the four operand layouts.
#define SDT_LAYOUTS_(X, ...) X(__VA_ARGS__, 0) X(__VA_ARGS__, 1) X(__VA_ARGS__, 2) X(__VA_ARGS__, 3)

#define SDT_PAIR_ONE_(BN, L)                                                                         \
    template int sdt::launch_gemm_pair<BN, L>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,   \
                                              const sdt::GemmArgs &, cudaStream_t);
#define SDT_INSTANTIATE_GEMM_PAIR(BN) SDT_LAYOUTS_(SDT_PAIR_ONE_, BN)

#define SDT_PERSISTENT_ONE_(BN, L)                                                                   \
    template int sdt::launch_gemm_persistent<BN, L>(const CUtensorMap &, const CUtensorMap &,        \
                                                    const CUtensorMap &, const sdt::GemmArgs &, cudaStream_t);
#define SDT_INSTANTIATE_GEMM_PERSISTENT(BN) SDT_LAYOUTS_(SDT_PERSISTENT_ONE_, BN)

#define SDT_TILE_ONE_(BM, BN, L)                                                                     \
    template int sdt::launch_gemm_tile<BM, BN, L>(const CUtensorMap &, const CUtensorMap &,          \
                                                  const CUtensorMap &, const sdt::GemmArgs &, cudaStream_t);
#define SDT_TILE_SPLIT_ONE_(BM, BN, L)                                                               \
    template int sdt::launch_gemm_tile_split<BM, BN, L>(const CUtensorMap &, const CUtensorMap &,    \
                                                        const sdt::GemmArgs &, cudaStream_t);
#define SDT_TILE_STREAM_ONE_(BM, BN, L)                                                              \
    template int sdt::launch_gemm_streamk<BM, BN, L>(const CUtensorMap &, const CUtensorMap &,       \
                                                     const sdt::GemmArgs &, cudaStream_t);
#define SDT_INSTANTIATE_GEMM_TILE(BM, BN)                                                            \
    SDT_LAYOUTS_(SDT_TILE_ONE_, BM, BN)                                                              \
    SDT_LAYOUTS_(SDT_TILE_SPLIT_ONE_, BM, BN)                                                        \
    SDT_LAYOUTS_(SDT_TILE_STREAM_ONE_, BM, BN)
