// gemm_noalloc.cu -- a split-K GEMM entry point that allocates nothing.
//
// gemm_f16_splitk needs a workspace for its fp32 partial tiles, and the
// library leaves allocating it to the caller.  Some callers cannot allocate
// device memory at the point where they multiply: code that must not
// synchronise the device (cudaMalloc and cudaFree can), plugin hosts that give
// a kernel library a fixed memory budget and no allocator, and latency-critical
// loops that forbid allocator calls altogether.  For them this entry point
// keeps the workspace in a file-scope __device__ array of fixed size, so a
// call only launches kernels.
//
// Set-up: in host code the array's name is only a host-side stand-in, never a
// device address, so on the first call on each device (with that device
// current) its device address is obtained once with cudaGetSymbolAddress and
// cached per device.  That first call should therefore come before any stream
// capture.
//
// Size: the workspace layout of gemm_f16_splitk puts a fixed 1 MiB region of
// arrival counters in front of the fp32 partials, so of the 16 MiB array
// 15 MiB hold partials: sdt_splitk_workspace_bytes (counters + partials) must
// be at most 16 MiB.  1024x1024 with 3 splits (12 MiB of partials), 512x512
// with 15 (15 MiB) and 256x256 with 32 (8 MiB) fit; 1024x1024 with 4 splits
// and 512x512 with 16 do not.  When the call picks the split count itself it
// lowers it until the partials fit, and refuses only a shape whose unsplit
// partials do not fit.
//
// Sharing: every call uses the same array and leaves its partials there.  The
// reduction algorithm used here (a separate summing kernel) overwrites every
// partial it later reads, so nothing in the array has to start at zero.  Calls
// whose executions overlap on the GPU (different streams, no ordering between
// them) race on the array and corrupt each other's results.
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.cuh"

namespace sdt {
int splitk_launch(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C, void *ws,
                  size_t ws_bytes, int tile_id, int splits, int algo, cudaStream_t stream);
}  // namespace sdt

using namespace sdt;

// 16 MiB: the 1 MiB counter region of the split-K workspace layout plus 15 MiB of fp32
// partials (e.g. 1024x1024 with 3 splits, 512x512 with 15).
static constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static constexpr int kNoAllocMaxDevices = 64;
static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[kNoAllocMaxDevices];

// Device address of the scratch array on the current device (looked up once per device).
static int noalloc_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        cudaGetLastError();
        return fail(SDT_ERR_UNSUPPORTED_DEVICE, "no usable CUDA device (%s)", cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return fail(SDT_ERR_CUDA, "cudaGetSymbolAddress of the no-allocation scratch failed on device %d: %s",
                        dev, cudaGetErrorString(e));
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SDT_OK;
}

extern "C" int gemm_f16_splitk_noalloc(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                                       int tile_id, int splits, sdt_stream_t stream) {
    clear_error();
    if (M < 0 || N < 0 || K < 0)
        return fail(SDT_ERR_SHAPE, "negative dimension (M=%lld N=%lld K=%lld)", (long long)M, (long long)N,
                    (long long)K);
    if (M == 0 || N == 0) return SDT_OK;
    void *scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // K == 0: the empty sum, C = 0, whatever the tile and split arguments (as gemm_f16_splitk)
    if (K == 0)
        return splitk_launch(M, N, K, A, B, C, scratch, kNoAllocScratchBytes, tile_id, splits,
                             SDT_SPLITK_REDUCE_KERNEL, s);
    if (tile_id < 0) {
        rc = sdt_device_sm_count();
        if (rc < 0) return rc;
        const int sm = rc;
        rc = sdt_device_smem_optin();
        if (rc < 0) return rc;
        int picked_splits = 1;
        rc = sdt_pick_splitk_for(M, N, K, sm, rc, &tile_id, &picked_splits);
        if (rc) return rc;
        if (splits <= 0) {
            // a split count the call chose is lowered until its partials fit the array
            splits = picked_splits;
            while (splits > 1 && sdt_splitk_workspace_bytes(M, N, K, tile_id, splits) > kNoAllocScratchBytes)
                --splits;
        }
    }
    const size_t need = sdt_splitk_workspace_bytes(M, N, K, tile_id, splits);
    if (need == 0)
        return fail(SDT_ERR_ARG, "tile %d with %d splits is not a valid split-K configuration for %lldx%lldx%lld",
                    tile_id, splits, (long long)M, (long long)N, (long long)K);
    if (need > kNoAllocScratchBytes)
        return fail(SDT_ERR_ARG,
                    "%lldx%lldx%lld with %d splits needs %zu bytes of scratch (1 MiB of counters + fp32 partials); "
                    "the fixed no-allocation scratch holds %zu bytes (use gemm_f16_splitk with a workspace, or "
                    "fewer splits)",
                    (long long)M, (long long)N, (long long)K, splits, need, kNoAllocScratchBytes);
    return splitk_launch(M, N, K, A, B, C, scratch, kNoAllocScratchBytes, tile_id, splits, SDT_SPLITK_REDUCE_KERNEL,
                         s);
}
