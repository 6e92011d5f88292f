// gemv.cu -- M = 1 decode: y[n] = sum_k x[k] * W[n][k], W stored K-major.
//
// "mojo-baro", section "Four rounds on the decode shape": the weight matrix has
// to stream out of HBM at close to full bandwidth; what decided speed there was
// coalescing (K-major weights, round v1), wide contiguous loads per thread
// (round v3) and an M=1-specialised kernel that keeps accumulators in registers
// (round v4); q8 (int8 with a scale per 32 weights, round v2) halves the bytes
// but only pays if dequantisation stays off the critical path.
//
// Two designs live here.  The default one (further down: gemv_q8_dp2a_kernel and
// gemv_bf16_rows_kernel) gives each CTA a balanced contiguous range of rows and
// its threads fixed 32-byte slices of every row, with the activations kept in
// registers, two batches of rows in flight, L2 prefetches that start before the
// previous kernel in the stream has finished, and q8 multiplied in int16 x int8
// dot products.  The first one, kept as a fallback for shapes the default does
// not take (K not a multiple of 16, K above 8192 for bf16 or 16384 for q8,
// weights only 16-byte aligned):
//
// One warp owns ROWS consecutive output rows at a time.  Lane l
// reads 16-byte chunks l, l+32, l+64, ... of each row, so every load instruction
// of the warp covers 512 contiguous bytes of one row.  U chunks per row are
// issued before any arithmetic so that ROWS*U 16-byte loads per lane are in
// flight.  Partial sums stay in fp32 registers and are combined with a
// butterfly of warp shuffles at the end of each row block.
//
//  bf16: a bf16 is the top half of an fp32, so conversion is a shift or a mask;
//        each product is exact in fp32 and is accumulated with packed (f32x2)
//        FMA into two partial sums per lane.
//  q8  : int8 weights are turned into exact fp32 values by placing the byte
//        (offset to unsigned) in the mantissa of 2^23 and subtracting 2^23+128
//        (packed f32x2 add); a 16-byte chunk is half of one 32-weight group, so
//        the group's fp16 scale multiplies the chunk's partial sum once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "host_common.cuh"
#include "launch.cuh"
#include "ptx.cuh"

namespace sdt {

__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}


__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Packed pairs of fp32 (sm_100-class f32x2 arithmetic): a 64-bit register holds
// two floats, low word first.
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ float sum2(uint64_t a) {
    return __uint_as_float(static_cast<uint32_t>(a)) + __uint_as_float(static_cast<uint32_t>(a >> 32));
}

// A bf16 pair word -> the two fp32 values, packed.
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) { return pack2(w << 16, w & 0xFFFF0000u); }

// Four int8 weights of one word (already xor-ed with 0x80808080, i.e. biased to
// unsigned) times four activations (two packed pairs), accumulated into a packed pair.
// Each byte u is placed in the mantissa of 2^23, so the float is exactly 2^23 + u;
// subtracting 2^23 + 128 gives the signed weight exactly.
__device__ __forceinline__ uint64_t dot4_q8(uint32_t qw, uint64_t x01, uint64_t x23, uint64_t acc) {
    const uint32_t magic = 0x4B000000u;                  // 2^23
    const uint32_t off = 0xCB000080u;                    // -(2^23 + 128)
    const uint64_t neg_off = pack2(off, off);
    const uint64_t q01 = add2(pack2(__byte_perm(qw, magic, 0x7540), __byte_perm(qw, magic, 0x7541)), neg_off);
    const uint64_t q23 = add2(pack2(__byte_perm(qw, magic, 0x7542), __byte_perm(qw, magic, 0x7543)), neg_off);
    acc = fma2(q01, x01, acc);
    acc = fma2(q23, x23, acc);
    return acc;
}

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;

// Eight bf16 weights times eight activations (packed pairs), accumulated into a packed pair.
__device__ __forceinline__ uint64_t dot8_bf16(const uint4 &w, const uint64_t (&xp)[4], uint64_t acc) {
    acc = fma2(bf16x2_to_f32x2(w.x), xp[0], acc);
    acc = fma2(bf16x2_to_f32x2(w.y), xp[1], acc);
    acc = fma2(bf16x2_to_f32x2(w.z), xp[2], acc);
    acc = fma2(bf16x2_to_f32x2(w.w), xp[3], acc);
    return acc;
}

template <int ROWS, int U>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_bf16_kernel(int K8, int N, const uint4 *__restrict__ x, const uint4 *__restrict__ W,
                     float *__restrict__ y) {
    griddep_launch_dependents();
    griddep_wait();  // x and W may come from the previous kernel
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * kGemvWarps;
    for (int n0 = gwarp * ROWS; n0 < N; n0 += nwarps * ROWS) {
        uint64_t acc[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) acc[r] = 0;
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
            for (int u = 0; u < U; ++u) {
                const uint64_t xp[4] = {bf16x2_to_f32x2(xv[u].x), bf16x2_to_f32x2(xv[u].y),
                                        bf16x2_to_f32x2(xv[u].z), bf16x2_to_f32x2(xv[u].w)};
#pragma unroll
                for (int r = 0; r < ROWS; ++r) acc[r] = dot8_bf16(w[r][u], xp, acc[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float v = warp_sum(sum2(acc[r]));
            if (lane == 0 && n0 + r < N) y[n0 + r] = v;
        }
    }
}

// K16 = K / 16 chunks of 16 int8 per row; scales [N][K/32] fp16.
template <int ROWS, int U>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_q8_kernel(int K16, int N, const uint4 *__restrict__ x, const uint4 *__restrict__ W,
                   const __half *__restrict__ scales, float *__restrict__ y) {
    griddep_launch_dependents();
    griddep_wait();  // x and W may come from the previous kernel
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
                // the chunk's 16 activations as 8 packed fp32 pairs, shared by the ROWS rows
                const uint64_t x0 = bf16x2_to_f32x2(xa.x), x1 = bf16x2_to_f32x2(xa.y);
                const uint64_t x2 = bf16x2_to_f32x2(xa.z), x3 = bf16x2_to_f32x2(xa.w);
                const uint64_t x4 = bf16x2_to_f32x2(xb.x), x5 = bf16x2_to_f32x2(xb.y);
                const uint64_t x6 = bf16x2_to_f32x2(xb.z), x7 = bf16x2_to_f32x2(xb.w);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    uint64_t part = 0;
                    part = dot4_q8(w[r][u].x ^ 0x80808080u, x0, x1, part);
                    part = dot4_q8(w[r][u].y ^ 0x80808080u, x2, x3, part);
                    part = dot4_q8(w[r][u].z ^ 0x80808080u, x4, x5, part);
                    part = dot4_q8(w[r][u].w ^ 0x80808080u, x6, x7, part);
                    acc[r] = fmaf(sc[r][u], sum2(part), acc[r]);
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

// ---------------------------------------------------------------------------------
// Streaming variant: weights (and q8 scales) staged through shared memory by bulk
// copies.
//
// One CTA per SM owns a contiguous slice of rows (a multiple of RS rows).  A
// producer thread streams the slice RS rows at a time -- one contiguous block of
// RS * row_bytes since W is row-major, plus the matching RS * K/16 bytes of q8
// scales -- into a ring of shared-memory stages with cp.async.bulk + mbarrier
// complete_tx, so the copy engine keeps many kilobytes in flight per SM
// independently of the consumers' arithmetic.  The activations are converted
// once per CTA to fp32 in shared memory.  NW consumer warps work on each stage:
// H warps per row (RS = NW / H rows), lane l of a warp reading 16-byte chunks
// h*32 + l, h*32 + l + 32*H, ... of its row, so all operands of the inner loop
// come from shared memory.  Partial sums stay in packed fp32 pairs; the H
// warps of a row combine through shared-memory atomics (no barrier between
// warps, so a warp that gives up a bounded wait cannot stall its partner).
// ---------------------------------------------------------------------------------

constexpr int kStreamConsumers = 16;
constexpr int kStreamThreads = (kStreamConsumers + 1) * 32;
constexpr int kStreamSmemBudget = 220 * 1024;

struct StreamArgs {
    const uint4 *x;        // bf16 activations [K]
    const uint8_t *W;      // [N][row_bytes]
    const uint8_t *scales; // q8: fp16 [N][K/32]
    float *y;
    int K, N;
    int row_bytes;
    int scale_row_bytes;   // q8: K/16; bf16: 0
    int stages;
    int rows_per_cta;      // multiple of the rows per stage
    unsigned long long timeout_ns;
    int *status;
};

template <bool Q8, int H>
__global__ void __launch_bounds__(kStreamThreads, 1) gemv_stream_kernel(const StreamArgs a) {
    constexpr int RS = kStreamConsumers / H;  // rows per stage
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 127u) & ~127u) - raw);
    const int S = a.stages;
    const int w_bytes = RS * a.row_bytes;
    const int sc_bytes = RS * a.scale_row_bytes;
    const int stage_bytes = w_bytes + sc_bytes;
    // Activations as fp32 pairs in a transposed layout: pair p of chunk c at xs2[p * nchunk + c],
    // so the 32 lanes of a warp (consecutive chunks) read 32 consecutive 8-byte words.
    uint2 *xs2 = reinterpret_cast<uint2 *>(smem + S * stage_bytes);  // K/2 pairs
    float *partial = reinterpret_cast<float *>(xs2 + (a.K >> 1));    // [S][RS] row sums (H > 1)
    uint32_t *arrived = reinterpret_cast<uint32_t *>(partial + S * RS);  // [S][RS] warps done
    uint64_t *full = reinterpret_cast<uint64_t *>(arrived + S * RS);
    uint64_t *empty = full + S;
    volatile uint32_t *ctrl = reinterpret_cast<volatile uint32_t *>(empty + S);  // [0] error, [1] issued

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r_begin = blockIdx.x * a.rows_per_cta;
    const int r_end = min(a.N, r_begin + a.rows_per_cta);
    const int n_st = r_end > r_begin ? (r_end - r_begin + RS - 1) / RS : 0;
    const uint64_t lim = a.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kStreamConsumers);
        }
        ctrl[0] = 0;
        ctrl[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();
    griddep_wait();  // x and W may come from the previous kernel

    if (warp == kStreamConsumers) {
        if (lane == 0) {
            int s = 0;
            uint32_t phase = 0;
            for (int st = 0; st < n_st; ++st) {
                if (!mbar_wait_for(smem_u32(&empty[s]), phase ^ 1u, lim)) {
                    if (a.status) atomicCAS(a.status, 0, static_cast<int>(kSiteProducer));
                    ctrl[0] = 1;
                    break;
                }
                if (ctrl[0]) break;
                const int r = r_begin + st * RS;
                const int nrows = min(RS, r_end - r);
                const uint32_t fb = smem_u32(&full[s]);
                uint8_t *dst = smem + s * stage_bytes;
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nrows * (a.row_bytes + a.scale_row_bytes)));
                bulk_load(smem_u32(dst), a.W + static_cast<size_t>(r) * a.row_bytes,
                          static_cast<uint32_t>(nrows * a.row_bytes), fb);
                if (Q8)
                    bulk_load(smem_u32(dst + w_bytes), a.scales + static_cast<size_t>(r) * a.scale_row_bytes,
                              static_cast<uint32_t>(nrows * a.scale_row_bytes), fb);
                ctrl[1] = static_cast<uint32_t>(st + 1);
                if (++s == S) { s = 0; phase ^= 1u; }
            }
        }
    } else {
        for (int i = threadIdx.x; i < S * RS; i += kStreamConsumers * 32) {
            partial[i] = 0.f;
            arrived[i] = 0u;
        }
        const int nchunk = a.K >> (Q8 ? 4 : 3);  // 16-byte weight chunks per row
        // activations -> fp32 pairs in shared memory (consumer warps only; the producer is
        // already streaming).  x word i holds elements 8i .. 8i+7: chunk 8i / E, pairs from
        // (8i % E) / 2, with E = 16 (q8) or 8 (bf16) elements per chunk.
        for (int i = threadIdx.x; i < (a.K >> 3); i += kStreamConsumers * 32) {
            const uint4 v = __ldg(a.x + i);
            const int c = Q8 ? (i >> 1) : i;
            const int p0 = Q8 ? (i & 1) * 4 : 0;
            xs2[(p0 + 0) * nchunk + c] = make_uint2(v.x << 16, v.x & 0xFFFF0000u);
            xs2[(p0 + 1) * nchunk + c] = make_uint2(v.y << 16, v.y & 0xFFFF0000u);
            xs2[(p0 + 2) * nchunk + c] = make_uint2(v.z << 16, v.z & 0xFFFF0000u);
            xs2[(p0 + 3) * nchunk + c] = make_uint2(v.w << 16, v.w & 0xFFFF0000u);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kStreamConsumers * 32) : "memory");

        const int row_in_stage = warp / H;
        const int h = warp % H;
        int s = 0;
        uint32_t phase = 0;
        for (int st = 0; st < n_st; ++st) {
            if (!warp_wait(smem_u32(&full[s]), phase, lim, lane)) {
                if (lane == 0) {
                    if (a.status) atomicCAS(a.status, 0, static_cast<int>(kSiteEpilogue));
                    ctrl[0] = 1;
                }
                break;
            }
            const int row = r_begin + st * RS + row_in_stage;
            const uint8_t *wrow = smem + s * stage_bytes + row_in_stage * a.row_bytes;
            const __half *srow = reinterpret_cast<const __half *>(smem + s * stage_bytes + w_bytes +
                                                                 row_in_stage * a.scale_row_bytes);
            float v = 0.f;
            if (row < r_end) {
                uint64_t acc = 0;
                float accf = 0.f;
#pragma unroll 4
                for (int c = h * 32 + lane; c < nchunk; c += 32 * H) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(wrow + c * 16);
                    if (Q8) {
                        const uint2 *xp = xs2 + c;
                        uint64_t part = 0;
                        const uint2 p0 = xp[0], p1 = xp[nchunk], p2 = xp[2 * nchunk], p3 = xp[3 * nchunk];
                        const uint2 p4 = xp[4 * nchunk], p5 = xp[5 * nchunk], p6 = xp[6 * nchunk],
                                    p7 = xp[7 * nchunk];
                        part = dot4_q8(w.x ^ 0x80808080u, pack2(p0.x, p0.y), pack2(p1.x, p1.y), part);
                        part = dot4_q8(w.y ^ 0x80808080u, pack2(p2.x, p2.y), pack2(p3.x, p3.y), part);
                        part = dot4_q8(w.z ^ 0x80808080u, pack2(p4.x, p4.y), pack2(p5.x, p5.y), part);
                        part = dot4_q8(w.w ^ 0x80808080u, pack2(p6.x, p6.y), pack2(p7.x, p7.y), part);
                        accf = fmaf(__half2float(srow[c >> 1]), sum2(part), accf);
                    } else {
                        const uint2 *xp = xs2 + c;
                        const uint2 p0 = xp[0], p1 = xp[nchunk], p2 = xp[2 * nchunk], p3 = xp[3 * nchunk];
                        acc = fma2(bf16x2_to_f32x2(w.x), pack2(p0.x, p0.y), acc);
                        acc = fma2(bf16x2_to_f32x2(w.y), pack2(p1.x, p1.y), acc);
                        acc = fma2(bf16x2_to_f32x2(w.z), pack2(p2.x, p2.y), acc);
                        acc = fma2(bf16x2_to_f32x2(w.w), pack2(p3.x, p3.y), acc);
                    }
                }
                v = warp_sum(Q8 ? accf : sum2(acc));
            }
            if (lane == 0) {
                if (H == 1) {
                    if (row < r_end) a.y[row] = v;
                } else {
                    // The H warps of a row add into the stage slot's sum; the last to arrive
                    // writes y and clears the slot.  The slot is reused only after this stage's
                    // empty barrier (which needs every warp's arrival below) has completed.
                    // With H = 2 the sum 0 + a + b is the same in either arrival order.
                    float *sum = &partial[s * RS + row_in_stage];
                    uint32_t *cnt = &arrived[s * RS + row_in_stage];
                    atomicAdd(sum, v);
                    __threadfence_block();
                    if (atomicAdd(cnt, 1u) == H - 1) {
                        __threadfence_block();
                        const float t = atomicExch(sum, 0.f);
                        atomicExch(cnt, 0u);
                        if (row < r_end) a.y[row] = t;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // this warp is done with the stage
            if (++s == S) { s = 0; phase ^= 1u; }
        }
    }

    __syncthreads();
    if (threadIdx.x == kStreamConsumers * 32 && ctrl[0]) {
        // drain: wait (bounded) for bulk copies this CTA issued and may not have seen land
        const int issued = static_cast<int>(ctrl[1]);
        for (int i = max(0, issued - S); i < issued; ++i)
            if (!mbar_wait_for(smem_u32(&full[i % S]), static_cast<uint32_t>((i / S) & 1), lim)) {
                if (a.status) atomicCAS(a.status, 0, static_cast<int>(kSiteDrain));
                break;
            }
    }
}

// ---------------------------------------------------------------------------------
// q8 on integer dot products (dp2a).
//
// The weights are integers, so the multiply-accumulate of a group of 32 can run
// in integer arithmetic once the activations are integers too.  Each group's 32
// activations are multiplied by the power of two 2^(14 - e) that puts the largest
// magnitude (binary exponent e) in [2^14, 2^15) and rounded to int16.  A bf16
// value within a factor 2^7 of the group's largest converts exactly (so do all
// integer inputs); a smaller one is off by at most 2^-15 of the group's largest.
// Then
//     y[n] = sum_g s[n,g] * 2^(e_g - 14) * sum_{k in g} xi[k] * q[n,k],
// where the inner sum is exact in int32 (|sum| < 32 * 2^15 * 2^7 = 2^27) and
// takes 16 dp2a instructions per group (each: two int16 x int8 products added
// to an int32), with no per-weight conversion at all.  The fp32 path above
// spends about four instructions per weight on conversion and packed FMA, and
// its byte permutes issue at a quarter of the FMA rate on this GPU, while dp2a
// issues at half rate: two per four weights.
//
// Work split: thread t of a CTA owns groups t, t + T, ... (GT of them) of every
// row, so its packed int16 activations stay in registers for the whole kernel.
// A CTA owns a contiguous, balanced range of rows and walks it RB rows at a time:
// one 32-byte load per row and group per thread (a warp reads 1 KB of one row per
// instruction), double-buffered so that the next RB rows are in flight while the
// current ones are summed.  Each row's partial sums are combined by a transposed
// butterfly within the warp and then across warps through shared memory, in a
// fixed order: results are deterministic.
//
// Launch-to-launch overlap: in a stream of decode kernels the device idles
// between the end of one kernel and the first loads of the next.  Each CTA
// therefore asks L2 for the first pf_bytes of its rows before waiting on the
// previous kernel (programmatic dependent launch lets it start as soon as an SM
// has room), and the kernel's own weight loads are marked evict-first in L2 so
// that its stream does not push those prefetched lines out.
constexpr int kDpMaxThreads = 256;

// Read-only 16-byte load kept in program order with the weight loads around it.
__device__ __forceinline__ uint4 ld_nc_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void ld_stream_v8(const uint8_t *p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                   "=r"(w[7])
                 : "l"(p));
}

// The same 32-byte load with an L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void ld_stream_v8_hint(const uint8_t *p, uint64_t pol, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                   "=r"(w[7])
                 : "l"(p), "l"(pol));
}

// c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo) or bytes 2, 3 (hi); all signed.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Sum RB per-lane values (one per row) over the warp.  Each round halves the
// values a lane holds: the lower lane of a pair keeps the lower half of the rows
// and receives its partner's copy of them, the upper lane the upper half.  After
// log2(RB) such rounds the remaining rounds are plain butterflies; lane l then
// holds the warp's sum for row l / (32 / RB).
template <int RB>
__device__ __forceinline__ float reduce_rows(float (&v)[RB], int lane) {
    int off = 16;
#pragma unroll
    for (int h = RB / 2; h >= 1; h /= 2) {
        const bool upper = lane & off;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? v[i] : v[i + h];
            const float keep = upper ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        off >>= 1;
    }
    float r = v[0];
#pragma unroll
    for (; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

template <int GT, int RB>
struct DpBatch {
    uint32_t w[RB][GT][8];  // 32 int8 weights per (row, group)
    uint16_t s[RB][GT];     // that group's scale (fp16 bits, converted where it is used)
};

// Read-only 2-byte load kept in program order with the weight loads, so that a
// batch's scales are requested with its weights and waited for only where they are
// used (a plain load converted on arrival would wait for its data where it is issued).
__device__ __forceinline__ uint16_t ld_nc_u16(const __half *p) {
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

template <bool EF, int GT, int RB>
__device__ __forceinline__ void dp_load(DpBatch<GT, RB> &b, int n0, int r_end, int K, int G, const int (&g)[GT],
                                        const uint8_t *__restrict__ W, const __half *__restrict__ scales,
                                        uint64_t pol) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int n = n0 + r;
#pragma unroll
        for (int i = 0; i < GT; ++i) {
            if (n < r_end && g[i] < G) {
                // (a run-time choice here would merge the two loads' registers and wait for each)
                if (EF) ld_stream_v8_hint(W + size_t(n) * K + size_t(g[i]) * 32, pol, b.w[r][i]);
                else ld_stream_v8(W + size_t(n) * K + size_t(g[i]) * 32, b.w[r][i]);
                b.s[r][i] = ld_nc_u16(scales + size_t(n) * G + g[i]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) b.w[r][i][j] = 0u;
                b.s[r][i] = 0;
            }
        }
    }
}

// Thread 0 asks L2 for rows [r0, r1) of W and of the scales (clipped to 16-byte
// boundaries inside the range).  These requests need no registers, so they add to
// the bytes in flight per SM beyond the two register batches; the branch on the
// thread index also keeps the compiler from sinking the batch loads issued just
// before it into the arithmetic that follows.
__device__ __forceinline__ void dp_prefetch_rows(int r0, int r1, int K, int G, const uint8_t *W,
                                                 const __half *scales) {
    if (threadIdx.x == 0 && r1 > r0) {
        const size_t w0 = size_t(r0) * K, wb = size_t(r1 - r0) * K;  // K % 32 == 0
        for (size_t o = 0; o < wb; o += 32768) bulk_prefetch_l2(W + w0 + o, uint32_t(wb - o < 32768 ? wb - o : 32768));
        const size_t s0 = (size_t(r0) * G * 2 + 15) & ~size_t(15), s1 = (size_t(r1) * G * 2) & ~size_t(15);
        if (s1 > s0 && (reinterpret_cast<uintptr_t>(scales) & 15) == 0)
            bulk_prefetch_l2(reinterpret_cast<const uint8_t *>(scales) + s0, uint32_t(s1 - s0));
    }
}

// The CTA's partial sums p[r] of rows n0 + r -> y: warp butterfly, then the warps'
// sums added in warp order by threads 0..RB-1 (one barrier; `red` alternates
// between two buffers by batch, so the next batch's writes cannot race the reads).
template <int RB>
__device__ __forceinline__ void store_warp_sums(float v, int n0, int r_end, float *red, float *__restrict__ y) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kLanesPerRow = 32 / RB;
    if (lane % kLanesPerRow == 0) red[warp * RB + lane / kLanesPerRow] = v;
    __syncthreads();
    if (int(threadIdx.x) < RB && n0 + int(threadIdx.x) < r_end) {
        float t = 0.f;
        for (int w = 0; w < int(blockDim.x >> 5); ++w) t += red[w * RB + threadIdx.x];
        y[n0 + threadIdx.x] = t;
    }
}

template <int RB>
__device__ __forceinline__ void store_rows(float (&p)[RB], int n0, int r_end, float *red, float *__restrict__ y) {
    store_warp_sums<RB>(reduce_rows<RB>(p, threadIdx.x & 31), n0, r_end, red, y);
}

template <int GT, int RB>
__device__ __forceinline__ void dp_dot(const DpBatch<GT, RB> &b, const uint32_t (&xi)[GT][16], const float (&xf)[GT],
                                       float (&p)[RB]) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        p[r] = 0.f;
#pragma unroll
        for (int i = 0; i < GT; ++i) {
            int acc = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                acc = dp2a_lo(xi[i][2 * j], b.w[r][i][j], acc);
                acc = dp2a_hi(xi[i][2 * j + 1], b.w[r][i][j], acc);
            }
            p[r] = fmaf(float(acc), __half2float(__ushort_as_half(b.s[r][i])) * xf[i], p[r]);
        }
    }
}

template <int GT, int RB, bool EF, int MINB = 1>
__global__ void __launch_bounds__(kDpMaxThreads, MINB)
    gemv_q8_dp2a_kernel(int K, int N, const uint4 *__restrict__ x, const uint8_t *__restrict__ W,
                        const __half *__restrict__ scales, float *__restrict__ y, uint32_t pf_bytes,
                        int ahead) {
    __shared__ float red[2][(kDpMaxThreads / 32) * RB];  // per-warp row sums, by batch parity
    griddep_launch_dependents();
    uint64_t pol = 0;
    if (EF) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    const int G = K >> 5;
    const int T = blockDim.x;
    const int r_begin = int(int64_t(N) * blockIdx.x / gridDim.x);
    const int r_end = int(int64_t(N) * (blockIdx.x + 1) / gridDim.x);
    int g[GT];
#pragma unroll
    for (int i = 0; i < GT; ++i) g[i] = threadIdx.x + i * T;
    if (pf_bytes && threadIdx.x == 0 && r_end > r_begin) {
        // Ask L2 for the first pf_bytes of this CTA's weight rows (and their scales) while
        // the previous kernel in the stream may still be running.  L2 is where global
        // memory is coherent, so a line fetched now and written by that kernel later is
        // updated in place: the loads after the wait below still see its results.
        const size_t slice = size_t(r_end - r_begin) * K;
        const size_t wb = slice < pf_bytes ? slice : size_t(pf_bytes);  // multiples of 16
        const uint8_t *wp = W + size_t(r_begin) * K;
        for (size_t o = 0; o < wb; o += 32768) bulk_prefetch_l2(wp + o, uint32_t(wb - o < 32768 ? wb - o : 32768));
        const size_t s0 = (size_t(r_begin) * G * 2 + 15) & ~size_t(15);  // inside this CTA's scale rows
        const size_t s1 = (size_t(r_begin) * G * 2 + (wb / K + 1) * G * 2) & ~size_t(15);
        const size_t s2 = (size_t(r_end) * G * 2) & ~size_t(15);
        const size_t s_end = s1 < s2 ? s1 : s2;
        const uint8_t *sp = reinterpret_cast<const uint8_t *>(scales);
        if (s_end > s0 && (reinterpret_cast<uintptr_t>(sp) & 15) == 0) bulk_prefetch_l2(sp + s0, uint32_t(s_end - s0));
    }
    griddep_wait();  // x and W may come from the previous kernel

    // Issue order: the activations first (an L2 hit, so they return while the weights
    // are still on their way), then the first two batches of weights, then the
    // conversion, which waits only for the activations.
    uint32_t xw[GT][16];
#pragma unroll
    for (int i = 0; i < GT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = g[i] < G ? ld_nc_v4(x + size_t(g[i]) * 4 + j) : make_uint4(0, 0, 0, 0);
            xw[i][4 * j] = v.x;
            xw[i][4 * j + 1] = v.y;
            xw[i][4 * j + 2] = v.z;
            xw[i][4 * j + 3] = v.w;
        }
    DpBatch<GT, RB> ba, bb;
    dp_load<EF>(ba, r_begin, r_end, K, G, g, W, scales, pol);
    dp_load<EF>(bb, r_begin + RB, r_end, K, G, g, W, scales, pol);
    // rows loaded into registers later are asked of L2 `ahead` rows in advance
    if (ahead) dp_prefetch_rows(r_begin + 2 * RB, min(r_begin + 2 * RB + ahead, r_end), K, G, W, scales);

    // this thread's groups of activations -> packed int16 pairs and the factor undoing the scaling
    uint32_t xi[GT][16];
    float xf[GT];
#pragma unroll
    for (int i = 0; i < GT; ++i) {
        uint32_t e2 = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) e2 = __vmaxu2(e2, xw[i][j] & 0x7F807F80u);  // exponent fields
        const uint32_t e_raw = max(e2 & 0xFFFFu, e2 >> 16) >> 7;
        // clamp tiny groups so both factors stay normal floats (values below 2^-111 are
        // rounded to multiples of 2^-125, far below any tolerance)
        const uint32_t e = max(e_raw, 16u);
        const float up = __uint_as_float((268u - e) << 23);  // 2^(14 - (e - 127))
        xf[i] = e_raw == 255u ? __uint_as_float(0x7FC00000u)  // Inf or NaN among the activations
                              : __uint_as_float((e - 14u) << 23);  // 2^((e - 127) - 14)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int lo = __float2int_rn(__uint_as_float(xw[i][j] << 16) * up);
            const int hi = __float2int_rn(__uint_as_float(xw[i][j] & 0xFFFF0000u) * up);
            xi[i][j] = (uint32_t(lo) & 0xFFFFu) | (uint32_t(hi) << 16);
        }
    }

    // batch pipeline: while one register set is summed, the other is in flight.  A
    // set's next rows are requested once its dot products are formed and summed within
    // the warp (one register per thread then holds them), before the cross-warp sum and
    // its barrier, so that two batches stay in flight through the sum.
    int n0 = r_begin, parity = 0;
    while (n0 < r_end) {
        float p[RB];
        dp_dot(ba, xi, xf, p);
        float v = reduce_rows<RB>(p, threadIdx.x & 31);
        if (n0 + 2 * RB < r_end) {
            dp_load<EF>(ba, n0 + 2 * RB, r_end, K, G, g, W, scales, pol);
            if (ahead) dp_prefetch_rows(n0 + 2 * RB + ahead, min(n0 + 3 * RB + ahead, r_end), K, G, W, scales);
        }
        store_warp_sums<RB>(v, n0, r_end, red[parity], y);
        parity ^= 1;
        if (n0 + RB >= r_end) break;
        dp_dot(bb, xi, xf, p);
        v = reduce_rows<RB>(p, threadIdx.x & 31);
        if (n0 + 3 * RB < r_end) {
            dp_load<EF>(bb, n0 + 3 * RB, r_end, K, G, g, W, scales, pol);
            if (ahead) dp_prefetch_rows(n0 + 3 * RB + ahead, min(n0 + 4 * RB + ahead, r_end), K, G, W, scales);
        }
        store_warp_sums<RB>(v, n0 + RB, r_end, red[parity], y);
        parity ^= 1;
        n0 += 2 * RB;
    }
}

// ---------------------------------------------------------------------------------
// bf16 decode on the same row-range skeleton.  Thread t owns the 32-byte units
// (16 weights) t, t + T, ... of every row and holds their activations in
// registers as fp32 pairs; per unit: one 32-byte load, 8 bf16 -> fp32 pair
// conversions (shift and mask) and 8 packed f32x2 FMAs.  Balanced row ranges,
// two register batches in flight, the L2 prefetch before the wait and one batch
// ahead, evict-first weight loads and the fixed-order reduction are as in the q8
// kernel above.
template <int GT, int RB>
struct BfBatch {
    uint32_t w[RB][GT][8];  // 16 bf16 weights per (row, unit)
};

template <bool EF, int GT, int RB>
__device__ __forceinline__ void bf_load(BfBatch<GT, RB> &b, int n0, int r_end, int K, int U, const int (&u)[GT],
                                        const uint8_t *__restrict__ W, uint64_t pol) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int n = n0 + r;
#pragma unroll
        for (int i = 0; i < GT; ++i) {
            if (n < r_end && u[i] < U) {
                const uint8_t *p = W + size_t(n) * 2 * K + size_t(u[i]) * 32;
                if (EF) ld_stream_v8_hint(p, pol, b.w[r][i]);
                else ld_stream_v8(p, b.w[r][i]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) b.w[r][i][j] = 0u;
            }
        }
    }
}

// Thread 0 asks L2 for rows [r0, r1) of a bf16 W (row bytes 2K, a multiple of 32).
__device__ __forceinline__ void bf_prefetch_rows(int r0, int r1, int K, const uint8_t *W) {
    if (threadIdx.x == 0 && r1 > r0) {
        const size_t w0 = size_t(r0) * 2 * K, wb = size_t(r1 - r0) * 2 * K;
        for (size_t o = 0; o < wb; o += 32768) bulk_prefetch_l2(W + w0 + o, uint32_t(wb - o < 32768 ? wb - o : 32768));
    }
}

// The CTA's partial sums of a batch's rows (one per thread and row) from its registers.
template <int GT, int RB>
__device__ __forceinline__ void bf_dot(const BfBatch<GT, RB> &b, const uint64_t (&xp)[GT][8], float (&p)[RB]) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        uint64_t acc = 0;
#pragma unroll
        for (int i = 0; i < GT; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc = fma2(bf16x2_to_f32x2(b.w[r][i][j]), xp[i][j], acc);
        p[r] = sum2(acc);
    }
}

template <int GT, int RB, bool EF, int MINB = 1>
__global__ void __launch_bounds__(kDpMaxThreads, MINB)
    gemv_bf16_rows_kernel(int K, int N, const uint4 *__restrict__ x, const uint8_t *__restrict__ W,
                          float *__restrict__ y, uint32_t pf_bytes, int ahead) {
    __shared__ float red[2][(kDpMaxThreads / 32) * RB];  // per-warp row sums, by batch parity
    griddep_launch_dependents();
    uint64_t pol = 0;
    if (EF) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    const int U = K >> 4;  // 32-byte units per row
    const int T = blockDim.x;
    const int r_begin = int(int64_t(N) * blockIdx.x / gridDim.x);
    const int r_end = int(int64_t(N) * (blockIdx.x + 1) / gridDim.x);
    int u[GT];
#pragma unroll
    for (int i = 0; i < GT; ++i) u[i] = threadIdx.x + i * T;
    if (pf_bytes && threadIdx.x == 0 && r_end > r_begin) {
        // as in the q8 kernel: only moves bytes of this CTA's rows into L2 early
        const size_t slice = size_t(r_end - r_begin) * 2 * K;
        const size_t wb = slice < pf_bytes ? slice : size_t(pf_bytes);
        const uint8_t *wp = W + size_t(r_begin) * 2 * K;
        for (size_t o = 0; o < wb; o += 32768) bulk_prefetch_l2(wp + o, uint32_t(wb - o < 32768 ? wb - o : 32768));
    }
    griddep_wait();  // x and W may come from the previous kernel

    uint32_t xw[GT][8];
#pragma unroll
    for (int i = 0; i < GT; ++i) {
        const uint4 v0 = u[i] < U ? ld_nc_v4(x + size_t(u[i]) * 2) : make_uint4(0, 0, 0, 0);
        const uint4 v1 = u[i] < U ? ld_nc_v4(x + size_t(u[i]) * 2 + 1) : make_uint4(0, 0, 0, 0);
        xw[i][0] = v0.x; xw[i][1] = v0.y; xw[i][2] = v0.z; xw[i][3] = v0.w;
        xw[i][4] = v1.x; xw[i][5] = v1.y; xw[i][6] = v1.z; xw[i][7] = v1.w;
    }
    BfBatch<GT, RB> ba, bb;
    bf_load<EF>(ba, r_begin, r_end, K, U, u, W, pol);
    bf_load<EF>(bb, r_begin + RB, r_end, K, U, u, W, pol);
    if (ahead) bf_prefetch_rows(r_begin + 2 * RB, min(r_begin + 2 * RB + ahead, r_end), K, W);
    uint64_t xp[GT][8];
#pragma unroll
    for (int i = 0; i < GT; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) xp[i][j] = bf16x2_to_f32x2(xw[i][j]);

    // A register set's next rows are requested as soon as its dot products are formed,
    // before the cross-warp sum and its barrier, so that two batches stay in flight
    // through the sum (2 % faster back to back on GB300 at K = 4096, N = 12288; the q8
    // kernel, at its 64-register cap, issues them after the warp's butterfly instead,
    // where its per-row partials have shrunk to one register).
    int n0 = r_begin, parity = 0;
    while (n0 < r_end) {
        float p[RB];
        bf_dot(ba, xp, p);
        if (n0 + 2 * RB < r_end) {
            bf_load<EF>(ba, n0 + 2 * RB, r_end, K, U, u, W, pol);
            if (ahead) bf_prefetch_rows(n0 + 2 * RB + ahead, min(n0 + 3 * RB + ahead, r_end), K, W);
        }
        store_rows<RB>(p, n0, r_end, red[parity], y);
        parity ^= 1;
        if (n0 + RB >= r_end) break;
        bf_dot(bb, xp, p);
        if (n0 + 3 * RB < r_end) {
            bf_load<EF>(bb, n0 + 3 * RB, r_end, K, U, u, W, pol);
            if (ahead) bf_prefetch_rows(n0 + 3 * RB + ahead, min(n0 + 4 * RB + ahead, r_end), K, W);
        }
        store_rows<RB>(p, n0 + RB, r_end, red[parity], y);
        parity ^= 1;
        n0 += 2 * RB;
    }
}

__global__ void zero_fill_f32(float *y, int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
        y[i] = 0.f;
}

// ---------------------------------------------------------------------------------
// Ring kernels (SDT_GEMV_VARIANT=ring).  One CTA per SM owns a
// balanced contiguous range of rows, which is one contiguous byte range of W (and
// of the q8 scales).  A producer thread streams that range through a ring of S
// shared-memory stages of RS rows with bulk copies (cp.async.bulk, completion on
// an mbarrier), so within the first microsecond of a launch every SM has S stages
// of its rows requested from HBM -- independently of the arithmetic and of any
// round trip -- and each stage is requested again as soon as it is consumed (the
// register kernels above keep at most two batches per thread in flight and refill
// them after a CTA-wide barrier per batch).  Measured on GB300 at K = 4096,
// N = 12288 it is the slower design: 17 us (q8) and 24 us (bf16) per launch back to
// back, against 8.3 and 15.2 us for the row-range kernels, and the same for rings of
// 60 to 200 KB -- one SM's bulk copies from HBM stay near 25 KB/us, below the
// ~45 KB/us that an SM's share of the HBM bandwidth needs, while plain loads from
// all of an SM's warps reach it.  It stays selectable for that comparison.
//
// Consumer thread t (of T) owns the 32-byte column slices t, t + T, ... of every row
// and keeps their activations in registers, as the row-range kernels do (q8: group-
// scaled int16 pairs for dp2a, bf16: packed fp32 pairs).  Per stage a warp sums its
// lanes' partials per row with the transposed butterfly and leaves one value per
// (row, warp) in shared memory, then every consumer lane arrives on the stage's
// "empty" barrier.  The producer, once that barrier completes, requests the next
// rows into the stage and then adds the stage's per-warp values in warp order (a
// fixed order: results are deterministic) and writes y.  The per-warp values are
// double-buffered by the stage's use count, so a refill cannot race the sum.
// ---------------------------------------------------------------------------------

struct RingArgs {
    const uint4 *x;          // bf16 activations [K]
    const uint8_t *W;        // [N][row_bytes]
    const uint8_t *scales;   // q8: fp16 [N][K/32]
    float *y;
    int K, N;
    int row_bytes;           // q8: K, bf16: 2K (a multiple of 32)
    int scale_row_bytes;     // q8: K/16 (a multiple of 16), bf16: 0
    int stages;
    uint32_t pf_bytes;       // W bytes of the CTA's range asked of L2 before the dependency wait
    int evict_first;         // weight copies marked evict-first in L2
    unsigned long long timeout_ns;
    int *status;
};

// cp.async.bulk global -> shared with an L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

template <bool Q8, int NCW, int GT, int RS>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) gemv_ring_kernel(const RingArgs a) {
    constexpr int T = NCW * 32;  // consumer threads
    static_assert(RS == 1 || RS == 2 || RS == 4 || RS == 8, "rows per stage: a power of two up to 8");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 127u) & ~127u) - raw);
    const int S = a.stages;
    const int w_bytes = RS * a.row_bytes;
    const int stage_bytes = w_bytes + RS * a.scale_row_bytes;  // a multiple of 16
    float *part = reinterpret_cast<float *>(smem + S * stage_bytes);  // [2][S][NCW][RS] per-warp row sums
    uint64_t *full = reinterpret_cast<uint64_t *>(part + 2 * S * NCW * RS);
    uint64_t *empty = full + S;
    volatile uint32_t *ctrl = reinterpret_cast<volatile uint32_t *>(empty + S);  // [0] gave up, [1] stages issued

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r_begin = int(int64_t(a.N) * blockIdx.x / gridDim.x);
    const int r_end = int(int64_t(a.N) * (blockIdx.x + 1) / gridDim.x);
    const int n_st = (r_end - r_begin + RS - 1) / RS;
    const uint64_t lim = a.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), T);
        }
        ctrl[0] = 0;
        ctrl[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();
    if (warp == NCW && lane == 0 && a.pf_bytes && r_end > r_begin) {
        // Ask L2 for the first pf_bytes of this CTA's rows while the previous kernel in the
        // stream may still run (L2 is the point of coherence: a line fetched now and written
        // by that kernel later is updated in place, and the copies after the wait see it).
        const size_t slice = size_t(r_end - r_begin) * a.row_bytes;
        const size_t wb = slice < a.pf_bytes ? slice : size_t(a.pf_bytes);  // multiples of 16
        const uint8_t *wp = a.W + size_t(r_begin) * a.row_bytes;
        for (size_t o = 0; o < wb; o += 32768) bulk_prefetch_l2(wp + o, uint32_t(wb - o < 32768 ? wb - o : 32768));
        if (Q8) {
            const size_t rows = wb / a.row_bytes + 1 < size_t(r_end - r_begin) ? wb / a.row_bytes + 1 : size_t(r_end - r_begin);
            bulk_prefetch_l2(a.scales + size_t(r_begin) * a.scale_row_bytes, uint32_t(rows * a.scale_row_bytes));
        }
    }
    griddep_wait();  // x and W may come from the previous kernel

    if (warp == NCW) {
        if (lane == 0) {
            // ---------------- producer: bulk copies into the ring, row sums out ----------------
            uint64_t pol = 0;
            if (a.evict_first) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
            const uint32_t ring0 = smem_u32(smem);
            // y rows of stage st (in slot s): the warps' values added in warp order
            auto finish = [&](int st, int s) {
                const int r0 = r_begin + st * RS;
                const int n = min(RS, r_end - r0);
                const float *pp = part + ((st / S) & 1) * S * NCW * RS + s * NCW * RS;
                for (int r = 0; r < n; ++r) {
                    float t = 0.f;
#pragma unroll
                    for (int w = 0; w < NCW; ++w) t += pp[w * RS + r];
                    a.y[r0 + r] = t;
                }
            };
            bool stop = false;
            for (int st = 0; st < n_st; ++st) {
                const int s = st % S;
                if (st >= S) {
                    // slot s last held stage st - S: every consumer lane must be done with it
                    if (!mbar_wait_for(empty0 + 8u * s, uint32_t((st / S - 1) & 1), lim)) {
                        if (a.status) atomicCAS(a.status, 0, static_cast<int>(kSiteProducer));
                        ctrl[0] = 1;
                        stop = true;
                        break;
                    }
                    if (ctrl[0]) { stop = true; break; }
                }
                const int r0 = r_begin + st * RS;
                const int n = min(RS, r_end - r0);
                const uint32_t fb = full0 + 8u * s;
                const uint32_t dst = ring0 + uint32_t(s * stage_bytes);
                mbar_arrive_expect_tx(fb, uint32_t(n * (a.row_bytes + a.scale_row_bytes)));
                const uint8_t *src = a.W + size_t(r0) * a.row_bytes;
                if (a.evict_first) bulk_load_hint(dst, src, uint32_t(n * a.row_bytes), fb, pol);
                else bulk_load(dst, src, uint32_t(n * a.row_bytes), fb);
                if (Q8)
                    bulk_load(dst + uint32_t(w_bytes), a.scales + size_t(r0) * a.scale_row_bytes,
                              uint32_t(n * a.scale_row_bytes), fb);
                ctrl[1] = uint32_t(st + 1);
                if (st >= S) finish(st - S, s);
            }
            // the stages still in the ring
            for (int st = max(0, n_st - S); st < n_st && !stop; ++st) {
                const int s = st % S;
                if (!mbar_wait_for(empty0 + 8u * s, uint32_t((st / S) & 1), lim)) {
                    if (a.status) atomicCAS(a.status, 0, static_cast<int>(kSiteProducer));
                    ctrl[0] = 1;
                    break;
                }
                finish(st, s);
            }
        }
    } else {
        // ---------------- consumers ----------------
        const int G = Q8 ? (a.K >> 5) : (a.K >> 4);  // 32-byte slices per row
        int g[GT];
#pragma unroll
        for (int i = 0; i < GT; ++i) g[i] = threadIdx.x + i * T;
        // activations of this thread's slices
        uint32_t xw[GT][Q8 ? 16 : 8];
#pragma unroll
        for (int i = 0; i < GT; ++i)
#pragma unroll
            for (int j = 0; j < (Q8 ? 4 : 2); ++j) {
                const uint4 v = g[i] < G ? ld_nc_v4(a.x + size_t(g[i]) * (Q8 ? 4 : 2) + j) : make_uint4(0, 0, 0, 0);
                xw[i][4 * j] = v.x;
                xw[i][4 * j + 1] = v.y;
                xw[i][4 * j + 2] = v.z;
                xw[i][4 * j + 3] = v.w;
            }
        // q8: group-scaled int16 pairs and the factor undoing the scaling (as gemv_q8_dp2a_kernel);
        // bf16: packed fp32 pairs
        uint32_t xi[GT][Q8 ? 16 : 1];
        float xf[GT];
        uint64_t xp[GT][Q8 ? 1 : 8];
#pragma unroll
        for (int i = 0; i < GT; ++i) {
            if constexpr (Q8) {
                uint32_t e2 = 0;
#pragma unroll
                for (int j = 0; j < 16; ++j) e2 = __vmaxu2(e2, xw[i][j] & 0x7F807F80u);
                const uint32_t e_raw = max(e2 & 0xFFFFu, e2 >> 16) >> 7;
                const uint32_t e = max(e_raw, 16u);
                const float up = __uint_as_float((268u - e) << 23);
                xf[i] = e_raw == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float((e - 14u) << 23);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int lo = __float2int_rn(__uint_as_float(xw[i][j] << 16) * up);
                    const int hi = __float2int_rn(__uint_as_float(xw[i][j] & 0xFFFF0000u) * up);
                    xi[i][j] = (uint32_t(lo) & 0xFFFFu) | (uint32_t(hi) << 16);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) xp[i][j] = bf16x2_to_f32x2(xw[i][j]);
            }
        }
        const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
        constexpr int kLanesPerRow = 32 / RS;
        for (int st = 0; st < n_st; ++st) {
            const int s = st % S;
            if (!warp_wait(full0 + 8u * s, uint32_t((st / S) & 1), lim, lane)) {
                if (lane == 0) {
                    if (a.status) atomicCAS(a.status, 0, static_cast<int>(kSiteEpilogue));
                    ctrl[0] = 1;
                }
                break;
            }
            const uint8_t *stage = smem + s * stage_bytes;
            float p[RS];
#pragma unroll
            for (int r = 0; r < RS; ++r) {
                const uint8_t *row = stage + r * a.row_bytes;
                if constexpr (Q8) {
                    const __half *sc = reinterpret_cast<const __half *>(stage + w_bytes + r * a.scale_row_bytes);
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < GT; ++i) {
                        if (g[i] < G) {
                            const uint4 w0 = *reinterpret_cast<const uint4 *>(row + g[i] * 32);
                            const uint4 w1 = *reinterpret_cast<const uint4 *>(row + g[i] * 32 + 16);
                            const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                            int d = 0;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                d = dp2a_lo(xi[i][2 * j], w[j], d);
                                d = dp2a_hi(xi[i][2 * j + 1], w[j], d);
                            }
                            acc = fmaf(float(d), __half2float(sc[g[i]]) * xf[i], acc);
                        }
                    }
                    p[r] = acc;
                } else {
                    uint64_t acc = 0;
#pragma unroll
                    for (int i = 0; i < GT; ++i) {
                        if (g[i] < G) {
                            const uint4 w0 = *reinterpret_cast<const uint4 *>(row + g[i] * 32);
                            const uint4 w1 = *reinterpret_cast<const uint4 *>(row + g[i] * 32 + 16);
                            acc = fma2(bf16x2_to_f32x2(w0.x), xp[i][0], acc);
                            acc = fma2(bf16x2_to_f32x2(w0.y), xp[i][1], acc);
                            acc = fma2(bf16x2_to_f32x2(w0.z), xp[i][2], acc);
                            acc = fma2(bf16x2_to_f32x2(w0.w), xp[i][3], acc);
                            acc = fma2(bf16x2_to_f32x2(w1.x), xp[i][4], acc);
                            acc = fma2(bf16x2_to_f32x2(w1.y), xp[i][5], acc);
                            acc = fma2(bf16x2_to_f32x2(w1.z), xp[i][6], acc);
                            acc = fma2(bf16x2_to_f32x2(w1.w), xp[i][7], acc);
                        }
                    }
                    p[r] = sum2(acc);
                }
            }
            const float v = reduce_rows<RS>(p, lane);
            if (lane % kLanesPerRow == 0)
                part[((st / S) & 1) * S * NCW * RS + s * NCW * RS + warp * RS + lane / kLanesPerRow] = v;
            mbar_arrive(empty0 + 8u * s);  // this lane is done with the stage (and its row sums are written)
        }
    }

    __syncthreads();
    if (threadIdx.x == NCW * 32 && ctrl[0]) {
        // drain: wait (bounded) for bulk copies this CTA issued and may not have seen land
        const int issued = static_cast<int>(ctrl[1]);
        for (int i = max(0, issued - S); i < issued; ++i)
            if (!mbar_wait_for(smem_u32(&full[i % S]), static_cast<uint32_t>((i / S) & 1), lim)) {
                if (a.status) atomicCAS(a.status, 0, static_cast<int>(kSiteDrain));
                break;
            }
    }
}

struct GemvVariant {
    int rows, unroll;  // register-path kernel: rows per warp, chunks in flight per row
    int stream_h;      // > 0: streaming kernel with this many consumer warps per row
    int rr_rows;       // > 0: the row-range kernel (q8: integer dot products) with this many rows per batch
    int ring;          // 1: the ring kernel first
};

// Variant selection.  Default: the row-range kernels with 2 rows per batch (q8 on
// integer dot products, bf16 on packed fp32 FMA) where their conditions hold, else
// the register kernel with 2 rows per warp and 4 chunks in flight per row.
// SDT_GEMV_VARIANT overrides: "ring" (the ring kernels first), "dp2" (row-range
// kernel, 2 rows per batch, either format), "dp4" / "dp8" (q8 integer kernel, rows
// per batch), "stream1" / "stream2" (streaming kernel, warps per row), "stream" (its
// default split), or "R,U" for the register kernel.
static GemvVariant gemv_variant(bool q8) {
    GemvVariant v{2, 4, 0, 2, 0};
    if (const char *s = getenv("SDT_GEMV_VARIANT")) {
        int r = 0, u = 0;
        if (!strcmp(s, "ring")) v.ring = 1;
        else if (!strcmp(s, "dp2")) v.ring = 0;
        else if (!strcmp(s, "dp4")) v = GemvVariant{2, 4, 0, q8 ? 4 : 0, 0};
        else if (!strcmp(s, "dp8")) v = GemvVariant{2, 4, 0, q8 ? 8 : 0, 0};
        else if (!strcmp(s, "stream1")) v = GemvVariant{2, 4, 1, 0, 0};
        else if (!strcmp(s, "stream2")) v = GemvVariant{2, 4, 2, 0, 0};
        else if (!strcmp(s, "stream")) v = GemvVariant{2, 4, q8 ? 1 : 2, 0, 0};
        else if (sscanf(s, "%d,%d", &r, &u) == 2) v = GemvVariant{r, u, 0, 0, 0};
    }
    return v;
}

// Shared memory the ring kernels give their ring (SDT_GEMV_RING_KB overrides), and
// the bytes of its rows each CTA asks L2 for before waiting on the previous kernel
// (SDT_GEMV_RING_PF_KB; 0 = none).
static int64_t gemv_ring_budget(int64_t default_kb) {
    int64_t kb = default_kb;
    if (const char *s = getenv("SDT_GEMV_RING_KB")) kb = std::max<long>(16, std::min<long>(strtol(s, nullptr, 10), 1024));
    return kb * 1024;
}
static uint32_t gemv_ring_prefetch(uint32_t default_kb) {
    long kb = default_kb;
    if (const char *s = getenv("SDT_GEMV_RING_PF_KB")) kb = std::max<long>(0, std::min<long>(strtol(s, nullptr, 10), 1 << 20));
    return uint32_t(kb) * 1024u;
}

template <bool Q8, int NCW, int GT, int RS>
static cudaError_t launch_ring(const RingArgs &a, int grid, int smem, cudaStream_t s, int device) {
    auto kern = gemv_ring_kernel<Q8, NCW, GT, RS>;
    static std::atomic<int> configured[64];
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (configured[device].load() < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[device].store(smem);
    }
    return launch_kernel(kern, dim3(grid), dim3((NCW + 1) * 32), size_t(smem), s, 1, a);
}

// The ring kernels take q8 with K % 256 == 0 (scale rows of whole 16-byte units),
// bf16 with K % 16 == 0 (whole 32-byte slices), up to 4 slices per consumer thread
// (K <= 16384), W and the scales 16-byte aligned (bulk copies), and a ring of at
// least two stages; returns false to ask for another kernel.  One CTA per SM:
// 4 consumer warps (q8, 4 rows per stage) or 8 (bf16, 2 rows per stage) and the
// producer warp.
static bool try_ring(bool q8, int64_t K, int64_t N, const void *x, const void *W, const void *scales, float *y,
                     cudaStream_t s, const DeviceInfo &dev, int *status, cudaError_t *err) {
    if (q8 ? (K % 256) : (K % 16)) return false;
    if ((reinterpret_cast<uintptr_t>(W) & 15) || (q8 && (reinterpret_cast<uintptr_t>(scales) & 15))) return false;
    const int ncw = q8 ? 4 : 8, rs = q8 ? 4 : 2;
    const int64_t T = int64_t(ncw) * 32;
    const int64_t slices = q8 ? K / 32 : K / 16;
    const int gt = slices <= T ? 1 : slices <= 2 * T ? 2 : slices <= 4 * T ? 4 : 0;
    if (gt == 0) return false;
    const int64_t row_bytes = q8 ? K : 2 * K;
    const int64_t scale_row_bytes = q8 ? K / 16 : 0;
    const int64_t stage_bytes = rs * (row_bytes + scale_row_bytes);
    const int64_t per_stage = stage_bytes + 8 * ncw * rs + 16;  // + the double-buffered row sums and two barriers
    const int64_t fixed = 128 + 8;
    const int64_t budget = std::min<int64_t>(gemv_ring_budget(200), dev.smem_optin);
    const int64_t stages = std::min<int64_t>((budget - fixed) / per_stage, 64);
    if (stages < 2) return false;
    RingArgs a;
    a.x = static_cast<const uint4 *>(x);
    a.W = static_cast<const uint8_t *>(W);
    a.scales = static_cast<const uint8_t *>(scales);
    a.y = y;
    a.K = int(K);
    a.N = int(N);
    a.row_bytes = int(row_bytes);
    a.scale_row_bytes = int(scale_row_bytes);
    a.stages = int(stages);
    a.pf_bytes = gemv_ring_prefetch(q8 ? 16 : 32);
    const char *ef_env = getenv("SDT_GEMV_EVICT_FIRST");
    a.evict_first = (ef_env && (!strcmp(ef_env, "0") || !strcmp(ef_env, "off"))) ? 0 : 1;
    a.timeout_ns = wait_timeout_ns();
    a.status = status;
    const int grid = int(std::min<int64_t>(dev.sm_count, N));
    const int smem = int(fixed + stages * per_stage);
    if (q8)
        *err = gt == 1 ? launch_ring<true, 4, 1, 4>(a, grid, smem, s, dev.device)
             : gt == 2 ? launch_ring<true, 4, 2, 4>(a, grid, smem, s, dev.device)
                       : launch_ring<true, 4, 4, 4>(a, grid, smem, s, dev.device);
    else
        *err = gt == 1 ? launch_ring<false, 8, 1, 2>(a, grid, smem, s, dev.device)
             : gt == 2 ? launch_ring<false, 8, 2, 2>(a, grid, smem, s, dev.device)
                       : launch_ring<false, 8, 4, 2>(a, grid, smem, s, dev.device);
    return true;
}

// Bytes of its weight rows each decode CTA asks L2 for before waiting on the
// previous kernel (SDT_GEMV_L2_PREFETCH_KB overrides; 0 turns the prefetch off).
// Measured best on GB300 at K=4096, N=12288: 12 KB (three rows) for q8, 32 KB (four
// rows) for bf16; larger prefetches compete with the previous kernel's last loads.
static uint32_t gemv_l2_prefetch_bytes(uint32_t default_kb) {
    if (const char *s = getenv("SDT_GEMV_L2_PREFETCH_KB")) {
        const long kb = strtol(s, nullptr, 10);
        return kb > 0 ? uint32_t(std::min<long>(kb, 1 << 20) * 1024) : 0u;
    }
    return default_kb * 1024;
}

// How many rows ahead of its register loads a decode CTA asks L2 for rows
// (SDT_GEMV_L2_AHEAD_ROWS, default one batch; rounded up to whole batches, 0 =
// none).  Measured on GB300 at K=4096, N=12288: one batch ahead is best; more
// only adds requests that compete with the register loads.
static int gemv_l2_ahead_rows(int rb) {
    int rows = rb;
    if (const char *s = getenv("SDT_GEMV_L2_AHEAD_ROWS")) rows = std::max(0, atoi(s));
    return (rows + rb - 1) / rb * rb;
}

// Launches the integer dot-product q8 kernel: T = ceil(G / GT) threads rounded up
// to a warp, one CTA per resident slot on every SM (balanced row ranges).
template <int GT, int RB, bool EF, int MINB = 1>
static cudaError_t launch_q8_dp(int K, int N, const void *x, const void *W, const void *sc, float *y,
                                cudaStream_t s, const DeviceInfo &dev) {
    auto kern = gemv_q8_dp2a_kernel<GT, RB, EF, MINB>;
    const int G = K / 32;
    const int T = ((G + GT - 1) / GT + 31) / 32 * 32;
    static std::atomic<int> occ_cache[64][kDpMaxThreads / 32];  // resident CTAs per SM, by device and T
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    std::atomic<int> &slot = occ_cache[dev.device][T / 32 - 1];
    int occ = slot.load();
    if (occ <= 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, T, 0);
        if (e != cudaSuccess) return e;
        if (occ < 1) occ = 1;
        slot.store(occ);
    }
    const int grid = int(std::min<int64_t>(int64_t(occ) * dev.sm_count, N));
    return launch_kernel(kern, dim3(grid), dim3(T), 0, s, 1, K, N, static_cast<const uint4 *>(x),
                         static_cast<const uint8_t *>(W), static_cast<const __half *>(sc), y,
                         gemv_l2_prefetch_bytes(12), gemv_l2_ahead_rows(RB));
}

// Launches the bf16 row-range kernel: T = ceil(U / GT) threads (U = K/16 units of
// 32 bytes per row) rounded up to a warp, one CTA per resident slot on every SM but
// ceil(SMs / 19) of them (8 on 152 SMs) left free: with every slot taken, a launch's
// CTAs can only become resident as the previous launch's leave; with a few free, some
// start at once and prefetch their first rows, and back-to-back launches ran 2.5 %
// faster on GB300 (K=4096, N=12288: 14.7-14.9 against 15.1-15.3 us on two boxes, any
// grid from 560 to 600 CTAs against 608).  The q8 kernel showed no such gain.
template <int GT, int RB, bool EF, int MINB>
static cudaError_t launch_bf16_rows(int K, int N, const void *x, const void *W, float *y, cudaStream_t s,
                                   const DeviceInfo &dev) {
    auto kern = gemv_bf16_rows_kernel<GT, RB, EF, MINB>;
    const int U = K / 16;
    const int T = ((U + GT - 1) / GT + 31) / 32 * 32;
    static std::atomic<int> occ_cache[64][kDpMaxThreads / 32];  // resident CTAs per SM, by device and T
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    std::atomic<int> &slot = occ_cache[dev.device][T / 32 - 1];
    int occ = slot.load();
    if (occ <= 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, T, 0);
        if (e != cudaSuccess) return e;
        if (occ < 1) occ = 1;
        slot.store(occ);
    }
    const int64_t slots = std::max<int64_t>(int64_t(occ) * dev.sm_count - (dev.sm_count + 18) / 19, 1);
    const int grid = int(std::min<int64_t>(slots, N));
    return launch_kernel(kern, dim3(grid), dim3(T), 0, s, 1, K, N, static_cast<const uint4 *>(x),
                         static_cast<const uint8_t *>(W), y, gemv_l2_prefetch_bytes(32), gemv_l2_ahead_rows(RB));
}

// The bf16 row-range kernel takes K % 16 == 0 (whole 32-byte units), K <= 8192
// (one or two units per thread) and 32-byte aligned weights; returns false to ask
// for another kernel.
static bool try_bf16_rows(int rows, int64_t K, int64_t N, const void *x, const void *W, float *y, cudaStream_t s,
                          const DeviceInfo &dev, cudaError_t *err) {
    if (rows != 2 || K % 16 || (reinterpret_cast<uintptr_t>(W) & 31)) return false;
    const char *ef_env = getenv("SDT_GEMV_EVICT_FIRST");
    const bool ef = !(ef_env && (!strcmp(ef_env, "0") || !strcmp(ef_env, "off")));
    const int64_t U = K / 16;
    const int k = int(K), n = int(N);
    if (U <= kDpMaxThreads) {
        *err = ef ? launch_bf16_rows<1, 2, true, 4>(k, n, x, W, y, s, dev)
                  : launch_bf16_rows<1, 2, false, 4>(k, n, x, W, y, s, dev);
        return true;
    }
    if (U <= 2 * kDpMaxThreads) {
        *err = ef ? launch_bf16_rows<2, 2, true, 2>(k, n, x, W, y, s, dev)
                  : launch_bf16_rows<2, 2, false, 2>(k, n, x, W, y, s, dev);
        return true;
    }
    return false;
}

// The integer kernel takes up to 256 threads of 1 or 2 groups each (K <= 16384)
// and 32-byte aligned weights (its loads are 32 bytes); returns false to ask for
// another kernel.  Two rows per batch with registers capped at 64 (8 CTAs of 128
// threads per SM) keeps the most bytes in flight and measured fastest; the weight
// loads are marked evict-first in L2 (SDT_GEMV_EVICT_FIRST=0 turns that off) so
// they do not displace the next kernel's prefetched rows.
static bool try_q8_dp(int rows, int64_t K, int64_t N, const void *x, const void *W, const void *scales, float *y,
                      cudaStream_t s, const DeviceInfo &dev, cudaError_t *err) {
    if (rows != 2 && rows != 4 && rows != 8) return false;
    if (reinterpret_cast<uintptr_t>(W) & 31) return false;
    const int64_t G = K / 32;
    const char *ef_env = getenv("SDT_GEMV_EVICT_FIRST");
    const bool ef = !(ef_env && (!strcmp(ef_env, "0") || !strcmp(ef_env, "off")));
    const int k = int(K), n = int(N);
    if (G <= kDpMaxThreads) {
        if (rows == 2)
            *err = ef ? launch_q8_dp<1, 2, true, 4>(k, n, x, W, scales, y, s, dev)
                      : launch_q8_dp<1, 2, false, 4>(k, n, x, W, scales, y, s, dev);
        else if (rows == 4)
            *err = ef ? launch_q8_dp<1, 4, true>(k, n, x, W, scales, y, s, dev)
                      : launch_q8_dp<1, 4, false>(k, n, x, W, scales, y, s, dev);
        else
            *err = ef ? launch_q8_dp<1, 8, true>(k, n, x, W, scales, y, s, dev)
                      : launch_q8_dp<1, 8, false>(k, n, x, W, scales, y, s, dev);
        return true;
    }
    if (G <= 2 * kDpMaxThreads) {
        *err = ef ? launch_q8_dp<2, 4, true>(k, n, x, W, scales, y, s, dev)
                  : launch_q8_dp<2, 4, false>(k, n, x, W, scales, y, s, dev);
        return true;
    }
    return false;
}

template <bool Q8, int H>
static cudaError_t launch_stream(const StreamArgs &a, int grid, int smem, cudaStream_t s) {
    auto kern = gemv_stream_kernel<Q8, H>;
    static std::atomic<int> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (configured[dev].load() < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev].store(smem);
    }
    return launch_kernel(kern, dim3(grid), dim3(kStreamThreads), size_t(smem), s, 1, a);
}

// Streams W through shared memory when a ring of at least two stages fits (with the
// fp32 activations); returns false to ask for the register kernel.
static bool try_stream(bool q8, int H, int64_t K, int64_t N, const void *x, const void *W, const void *scales,
                       float *y, cudaStream_t s, const DeviceInfo &dev, int *status, cudaError_t *err) {
    if (H != 1 && H != 2) return false;
    // every bulk copy must be a multiple of 16 bytes: q8 scale rows (K/16 bytes) need K % 256 == 0
    if (q8 && K % 256) return false;
    const int64_t RS = kStreamConsumers / H;
    const int64_t row_bytes = q8 ? K : 2 * K;
    const int64_t scale_row_bytes = q8 ? K / 16 : 0;
    const int64_t stage_bytes = RS * (row_bytes + scale_row_bytes);
    // per stage: the weights + scales, two 8-byte barriers, RS row sums and RS counters
    const int64_t per_stage = stage_bytes + 16 + 8 * RS;
    const int64_t fixed = 128 + 4 * K + 8;
    const int64_t budget = std::min<int64_t>(kStreamSmemBudget, dev.smem_optin);
    int64_t stages = (budget - fixed) / per_stage;
    if (stages > 8) stages = 8;
    if (stages < 2) return false;
    const int64_t min_rows = RS;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(dev.sm_count, (N + min_rows - 1) / min_rows));
    int64_t rows_per_cta = (N + grid - 1) / grid;
    rows_per_cta = (rows_per_cta + RS - 1) / RS * RS;  // whole stages (16-byte aligned scale copies)
    const int64_t ctas = (N + rows_per_cta - 1) / rows_per_cta;
    StreamArgs a;
    a.x = static_cast<const uint4 *>(x);
    a.W = static_cast<const uint8_t *>(W);
    a.scales = static_cast<const uint8_t *>(scales);
    a.y = y;
    a.K = int(K);
    a.N = int(N);
    a.row_bytes = int(row_bytes);
    a.scale_row_bytes = int(scale_row_bytes);
    a.stages = int(stages);
    a.rows_per_cta = int(rows_per_cta);
    a.timeout_ns = wait_timeout_ns();
    a.status = status;
    const int smem = int(fixed + stages * per_stage);
    if (q8) *err = H == 1 ? launch_stream<true, 1>(a, int(ctas), smem, s) : launch_stream<true, 2>(a, int(ctas), smem, s);
    else *err = H == 1 ? launch_stream<false, 1>(a, int(ctas), smem, s) : launch_stream<false, 2>(a, int(ctas), smem, s);
    return true;
}

template <int R, int U>
static cudaError_t launch_bf16(int K8, int N, const void *x, const void *W, float *y, cudaStream_t s) {
    const int rows_per_block = kGemvWarps * R;
    const int blocks = (N + rows_per_block - 1) / rows_per_block;
    return launch_kernel(gemv_bf16_kernel<R, U>, dim3(blocks), dim3(kGemvThreads), 0, s, 1, K8, N,
                  static_cast<const uint4 *>(x), static_cast<const uint4 *>(W), y);
}

template <int R, int U>
static cudaError_t launch_q8(int K16, int N, const void *x, const void *W, const void *sc, float *y,
                             cudaStream_t s) {
    const int rows_per_block = kGemvWarps * R;
    const int blocks = (N + rows_per_block - 1) / rows_per_block;
    return launch_kernel(gemv_q8_kernel<R, U>, dim3(blocks), dim3(kGemvThreads), 0, s, 1, K16, N,
                  static_cast<const uint4 *>(x), static_cast<const uint4 *>(W), static_cast<const __half *>(sc), y);
}

#define SDT_GEMV_DISPATCH(E, FN, V, ...)                                                           \
    do {                                                                                           \
        if (V.rows == 1 && V.unroll == 4) E = FN<1, 4>(__VA_ARGS__);                               \
        else if (V.rows == 1 && V.unroll == 8) E = FN<1, 8>(__VA_ARGS__);                          \
        else if (V.rows == 2 && V.unroll == 2) E = FN<2, 2>(__VA_ARGS__);                          \
        else if (V.rows == 4 && V.unroll == 2) E = FN<4, 2>(__VA_ARGS__);                          \
        else if (V.rows == 4 && V.unroll == 4) E = FN<4, 4>(__VA_ARGS__);                          \
        else E = FN<2, 4>(__VA_ARGS__);                                                            \
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
    cudaError_t e = cudaSuccess;
    if (K == 0) {
        const int blocks = int(std::min<int64_t>((N + 255) / 256, int64_t(dev.sm_count) * 4));
        zero_fill_f32<<<blocks, 256, 0, s>>>(y, N);
        e = cudaGetLastError();
    } else {
        const GemvVariant v = gemv_variant(q8);
        int *status = nullptr;
        rc = status_word(&status);
        if (rc) return rc;
        if (!(v.ring && try_ring(q8, K, N, x, W, scales, y, s, dev, status, &e)) &&
            !(q8 && try_q8_dp(v.rr_rows, K, N, x, W, scales, y, s, dev, &e)) &&
            !(!q8 && try_bf16_rows(v.rr_rows, K, N, x, W, y, s, dev, &e)) &&
            !try_stream(q8, v.stream_h, K, N, x, W, scales, y, s, dev, status, &e)) {
            if (!q8) SDT_GEMV_DISPATCH(e, launch_bf16, v, int(K / 8), int(N), x, W, y, s);
            else SDT_GEMV_DISPATCH(e, launch_q8, v, int(K / 16), int(N), x, W, scales, y, s);
        }
    }
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
