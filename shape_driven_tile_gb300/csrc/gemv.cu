// gemv.cu -- M = 1 decode: y[n] = sum_k x[k] * W[n][k], W stored K-major.
//
// "mojo-baro", section "Four rounds on the decode shape": the weight matrix has
// to stream out of HBM at close to full bandwidth; what decided speed there was
// coalescing (K-major weights, round v1), wide contiguous loads per thread
// (round v3) and an M=1-specialised kernel that keeps accumulators in registers
// (round v4); q8 (int8 with a scale per 32 weights, round v2) halves the bytes
// but only pays if dequantisation stays off the critical path.
//
// Design here: one warp owns ROWS consecutive output rows at a time.  Lane l
// reads 16-byte chunks l, l+32, l+64, ... of each row, so every load instruction
// of the warp covers 512 contiguous bytes of one row.  U chunks per row are
// issued before any arithmetic so that ROWS*U 16-byte loads per lane are in
// flight.  Partial sums stay in fp32 registers and are combined with a
// butterfly of warp shuffles at the end of each row block.
//
//  bf16: a bf16 is the top half of an fp32, so conversion is a shift or a mask;
//        each product is exact in fp32 and is accumulated with FMA.
//  q8  : int8 weights are turned into exact fp32 values by placing the byte
//        (offset to unsigned) in the mantissa of 2^23 and subtracting 2^23+128;
//        a 16-byte chunk is half of one 32-weight group, so the group's fp16
//        scale multiplies the chunk's partial sum once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "host_common.cuh"

namespace sdt {

__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float dot8_bf16(const uint4 &w, const uint4 &x, float acc) {
    acc = fmaf(bf16_lo(w.x), bf16_lo(x.x), acc);
    acc = fmaf(bf16_hi(w.x), bf16_hi(x.x), acc);
    acc = fmaf(bf16_lo(w.y), bf16_lo(x.y), acc);
    acc = fmaf(bf16_hi(w.y), bf16_hi(x.y), acc);
    acc = fmaf(bf16_lo(w.z), bf16_lo(x.z), acc);
    acc = fmaf(bf16_hi(w.z), bf16_hi(x.z), acc);
    acc = fmaf(bf16_lo(w.w), bf16_lo(x.w), acc);
    acc = fmaf(bf16_hi(w.w), bf16_hi(x.w), acc);
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Four int8 weights of one 32-bit word (already xor-ed with 0x80808080) times four
// bf16 activations (two words), accumulated into acc.
__device__ __forceinline__ float dot4_q8(uint32_t qw, uint32_t x01, uint32_t x23, float acc) {
    const uint32_t magic = 0x4B000000u;  // 2^23
    const float off = 8388736.0f;        // 2^23 + 128
    const float q0 = __uint_as_float(__byte_perm(qw, magic, 0x7540)) - off;
    const float q1 = __uint_as_float(__byte_perm(qw, magic, 0x7541)) - off;
    const float q2 = __uint_as_float(__byte_perm(qw, magic, 0x7542)) - off;
    const float q3 = __uint_as_float(__byte_perm(qw, magic, 0x7543)) - off;
    acc = fmaf(q0, bf16_lo(x01), acc);
    acc = fmaf(q1, bf16_hi(x01), acc);
    acc = fmaf(q2, bf16_lo(x23), acc);
    acc = fmaf(q3, bf16_hi(x23), acc);
    return acc;
}

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;

template <int ROWS, int U>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_bf16_kernel(int K8, int N, const uint4 *__restrict__ x, const uint4 *__restrict__ W,
                     float *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * kGemvWarps;
    for (int n0 = gwarp * ROWS; n0 < N; n0 += nwarps * ROWS) {
        float acc[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) acc[r] = 0.f;
        for (int c0 = lane; c0 < K8; c0 += 32 * U) {
            uint4 w[ROWS][U];
            uint4 xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
                const bool in = c < K8;
#pragma unroll
                for (int r = 0; r < ROWS; ++r)
                    w[r][u] = (in && n0 + r < N) ? ld_stream_v4(W + size_t(n0 + r) * K8 + c)
                                                 : make_uint4(0, 0, 0, 0);
                xv[u] = in ? __ldg(x + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < ROWS; ++r) acc[r] = dot8_bf16(w[r][u], xv[u], acc[r]);
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float v = warp_sum(acc[r]);
            if (lane == 0 && n0 + r < N) y[n0 + r] = v;
        }
    }
}

// K16 = K / 16 chunks of 16 int8 per row; scales [N][K/32] fp16.
template <int ROWS, int U>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_q8_kernel(int K16, int N, const uint4 *__restrict__ x, const uint4 *__restrict__ W,
                   const __half *__restrict__ scales, float *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * kGemvWarps;
    const int G = K16 >> 1;  // groups per row
    for (int n0 = gwarp * ROWS; n0 < N; n0 += nwarps * ROWS) {
        float acc[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) acc[r] = 0.f;
        for (int c0 = lane; c0 < K16; c0 += 32 * U) {
            uint4 w[ROWS][U];
            float sc[ROWS][U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
                const bool in = c < K16;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const bool ok = in && n0 + r < N;
                    w[r][u] = ok ? ld_stream_v4(W + size_t(n0 + r) * K16 + c) : make_uint4(0, 0, 0, 0);
                    sc[r][u] = ok ? __half2float(scales[size_t(n0 + r) * G + (c >> 1)]) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
                const bool in = c < K16;
                const uint4 xa = in ? __ldg(x + 2 * c) : make_uint4(0, 0, 0, 0);
                const uint4 xb = in ? __ldg(x + 2 * c + 1) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint4 q = make_uint4(w[r][u].x ^ 0x80808080u, w[r][u].y ^ 0x80808080u,
                                               w[r][u].z ^ 0x80808080u, w[r][u].w ^ 0x80808080u);
                    float part = 0.f;
                    part = dot4_q8(q.x, xa.x, xa.y, part);
                    part = dot4_q8(q.y, xa.z, xa.w, part);
                    part = dot4_q8(q.z, xb.x, xb.y, part);
                    part = dot4_q8(q.w, xb.z, xb.w, part);
                    acc[r] = fmaf(sc[r][u], part, acc[r]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float v = warp_sum(acc[r]);
            if (lane == 0 && n0 + r < N) y[n0 + r] = v;
        }
    }
}

__global__ void zero_fill_f32(float *y, int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
        y[i] = 0.f;
}

struct GemvVariant {
    int rows, unroll;
};

// Variant selection (rows per warp, chunks in flight per row); SDT_GEMV_VARIANT="R,U" overrides.
static GemvVariant gemv_variant(bool q8) {
    GemvVariant v = q8 ? GemvVariant{2, 4} : GemvVariant{2, 4};
    if (const char *s = getenv("SDT_GEMV_VARIANT")) {
        int r = 0, u = 0;
        if (sscanf(s, "%d,%d", &r, &u) == 2) v = GemvVariant{r, u};
    }
    return v;
}

template <int R, int U>
static void launch_bf16(int K8, int N, const void *x, const void *W, float *y, cudaStream_t s) {
    const int rows_per_block = kGemvWarps * R;
    const int blocks = (N + rows_per_block - 1) / rows_per_block;
    gemv_bf16_kernel<R, U><<<blocks, kGemvThreads, 0, s>>>(K8, N, static_cast<const uint4 *>(x),
                                                            static_cast<const uint4 *>(W), y);
}

template <int R, int U>
static void launch_q8(int K16, int N, const void *x, const void *W, const void *sc, float *y,
                      cudaStream_t s) {
    const int rows_per_block = kGemvWarps * R;
    const int blocks = (N + rows_per_block - 1) / rows_per_block;
    gemv_q8_kernel<R, U><<<blocks, kGemvThreads, 0, s>>>(K16, N, static_cast<const uint4 *>(x),
                                                          static_cast<const uint4 *>(W),
                                                          static_cast<const __half *>(sc), y);
}

#define SDT_GEMV_DISPATCH(FN, V, ...)                                                              \
    do {                                                                                           \
        if (V.rows == 1 && V.unroll == 4) FN<1, 4>(__VA_ARGS__);                                   \
        else if (V.rows == 1 && V.unroll == 8) FN<1, 8>(__VA_ARGS__);                              \
        else if (V.rows == 2 && V.unroll == 2) FN<2, 2>(__VA_ARGS__);                              \
        else if (V.rows == 4 && V.unroll == 2) FN<4, 2>(__VA_ARGS__);                              \
        else if (V.rows == 4 && V.unroll == 4) FN<4, 4>(__VA_ARGS__);                              \
        else FN<2, 4>(__VA_ARGS__);                                                                \
    } while (0)

static constexpr int64_t kGemvMaxDim = int64_t(1) << 30;

static int gemv_impl(int64_t K, int64_t N, const void *x, const void *W, const void *scales, float *y,
                     sdt_stream_t stream_h, bool q8) {
    clear_error();
    if (K < 0 || N < 0) return fail(SDT_ERR_SHAPE, "negative dimension");
    if (N == 0) return SDT_OK;
    if (K > kGemvMaxDim || N > kGemvMaxDim) return fail(SDT_ERR_SHAPE, "dimension too large");
    if (!y || (K > 0 && (!x || !W || (q8 && !scales)))) return fail(SDT_ERR_NULL, "NULL operand pointer");
    if ((reinterpret_cast<uintptr_t>(y) & 15) ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(W) & 15))))
        return fail(SDT_ERR_ALIGN, "x, W and y must be 16-byte aligned");
    if (q8 && K > 0 && (reinterpret_cast<uintptr_t>(scales) & 1))
        return fail(SDT_ERR_ALIGN, "scales must be 2-byte aligned");
    if (!q8 && K % 8) return fail(SDT_ERR_SHAPE, "bf16 gemv needs K %% 8 == 0 (K=%lld)", (long long)K);
    if (q8 && K % 32) return fail(SDT_ERR_SHAPE, "q8 gemv needs K %% 32 == 0 (K=%lld)", (long long)K);
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_h);
    if (K == 0) {
        const int blocks = int(std::min<int64_t>((N + 255) / 256, int64_t(dev.sm_count) * 4));
        zero_fill_f32<<<blocks, 256, 0, s>>>(y, N);
    } else if (!q8) {
        const GemvVariant v = gemv_variant(false);
        SDT_GEMV_DISPATCH(launch_bf16, v, int(K / 8), int(N), x, W, y, s);
    } else {
        const GemvVariant v = gemv_variant(true);
        SDT_GEMV_DISPATCH(launch_q8, v, int(K / 16), int(N), x, W, scales, y, s);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SDT_ERR_LAUNCH, "gemv launch failed: %s", cudaGetErrorString(e));
    return SDT_OK;
}

}  // namespace sdt

using namespace sdt;

extern "C" {

int gemv_m1(int64_t K, int64_t N, const void *x, const void *W, const void *scales, float *y,
            sdt_stream_t stream) {
    return gemv_impl(K, N, x, W, scales, y, stream, scales != nullptr);
}

int gemv_m1_bf16(int64_t K, int64_t N, const void *x, const void *W, float *y, sdt_stream_t stream) {
    return gemv_impl(K, N, x, W, nullptr, y, stream, false);
}

int gemv_m1_q8(int64_t K, int64_t N, const void *x, const void *W, const void *scales, float *y,
               sdt_stream_t stream) {
    return gemv_impl(K, N, x, W, scales, y, stream, true);
}

}  // extern "C"
