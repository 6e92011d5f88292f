// gemm_streamk.cuh -- stream-K form of the one-CTA ladder tiles.
//
// "Iteratively Tuning hipBLASLt TensileLite Kernels", section "The Six Rounds",
// the last round ("Stream-K"): instead of splitting K into equal slices per output
// tile, a fixed grid of workgroups shares the whole iteration space, so the work is
// spread evenly whatever the tile count; a workgroup's share may end part-way
// through an output tile, and the partial tiles are fixed up afterwards.  Here the iteration space is
// the list of (output tile, 64-deep k-tile) units, tiles in banded raster order
// and k-tiles in order within a tile; CTA g of G owns the contiguous units
// [floor(g*U/G), floor((g+1)*U/G)), so every CTA gets the same number of k-tiles
// to within one whatever the tile count, and a grid of one CTA per SM has no
// partial last wave.
//
// A CTA walks its units as segments (one per output tile it touches).  A segment
// that covers a whole tile is stored to C directly.  A segment that covers part
// of a tile is written as an fp32 partial tile to the CTA's slot in the
// workspace -- slot 2g for the CTA's first tile, 2g+1 for its last (every tile in
// between is whole) -- and then, per TMEM lane quarter, the epilogue warp counts
// its arrival on the tile's counter; the warp that arrives last sums the
// partials of all the tile's CTAs in CTA order (so the result does not depend on
// the order of arrival), rounds once to fp16/bf16, writes C and resets the counter
// to zero.  No CTA ever waits for another one.  Alternatively (splitk_reduce_in_kernel
// = 0) the kernel only writes the partials and a second kernel sums every shared
// tile with the whole GPU, in the same order (streamk_reduce_kernel).
//
// Roles (192 threads, as the persistent kernel):
//   warp 0 lane 0 : TMA producer (ring slots: full/empty mbarriers)
//   warp 1        : TMEM allocation; lane 0 issues tcgen05.mma and commits
//   warps 2..5    : epilogue; warp w reads TMEM lane quarter w % 4
// The accumulator is double-buffered in TMEM (acc_full / acc_empty per buffer),
// so the epilogue of one segment overlaps the MMAs of the next.
//
// Every wait is bounded per wait; on expiry the kernel records the site in the
// status word and unwinds (producer stops, MMA warp waits for its own MMAs, TMA
// copies in flight are drained, TMEM is freed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_kernel.cuh"
#include "gemm_persistent.cuh"
#include "ptx.cuh"

namespace sdt {

template <int BM, int BN>
struct StreamCfg {
    static constexpr int A_BYTES = BM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators of BN columns
    static constexpr int THREADS = 192;
    static constexpr int EPI_WARPS = 4;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int CTRL_BYTES = 512;
    __host__ __device__ static constexpr int smem_bytes(int stages) {
        return ALIGN_SLACK + stages * STAGE_BYTES + CTRL_BYTES;
    }
    static_assert(BM == 64 || BM == 128, "BM must be 64 or 128");
    static_assert(BN == 16 || BN == 32 || BN == 64 || BN == 128 || BN == 256, "BN must be 16 .. 256");
    static_assert(TMEM_COLS <= 512, "two accumulators must fit in TMEM");
};

// First unit of CTA g when G CTAs share U units: floor(g * U / G).
__host__ __device__ __forceinline__ long long sk_first_unit(long long g, long long G, long long U) {
    return g * U / G;
}
// The CTA that owns unit u: the largest g with sk_first_unit(g) <= u.
__host__ __device__ __forceinline__ int sk_owner(long long u, long long G, long long U) {
    return static_cast<int>(((u + 1) * G - 1) / U);
}

// One segment of a CTA's units: output tile `tile`, k-tiles [kb, ke).  sk_next returns
// the segment that starts at unit u and advances u past it (u_end: the CTA's end).
struct SkSegment {
    int tile, kb, ke;
};
__device__ __forceinline__ SkSegment sk_next(long long &u, long long u_end, long long nK) {
    SkSegment sg;
    sg.tile = static_cast<int>(u / nK);
    sg.kb = static_cast<int>(u - static_cast<long long>(sg.tile) * nK);
    sg.ke = static_cast<int>(nK - sg.kb < u_end - u ? nK : sg.kb + (u_end - u));
    u += sg.ke - sg.kb;
    return sg;
}

// Eight fp32 values of problem row `row`, columns n0+c .. n0+c+7, into C (fp16/bf16):
// one 16-byte store into row `row` of C, or, for swapped operands, eight 2-byte
// stores down column `row` of C.  Columns at or beyond N are skipped.
__device__ __forceinline__ void sk_store8(const GemmArgs &p, int row, int col, const float4 &a, const float4 &b,
                                          bool bf16) {
    uint16_t *C = reinterpret_cast<uint16_t *>(p.C);
    if (p.c_trans) {
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int t = 0; t < 8; ++t)
            if (col + t < p.N) C[static_cast<size_t>(col + t) * p.ldc + row] = f32_to_16(v[t], bf16);
    } else if (col + 8 <= p.N) {  // N % 8 == 0 unless swapped
        *reinterpret_cast<uint4 *>(C + static_cast<size_t>(row) * p.ldc + col) = pack8_f32(a, b, bf16);
    }
}

template <int BM, int BN, int LAYOUT>
__global__ void __launch_bounds__(192, 1)
    gemm_streamk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs p) {
    using Cfg = StreamCfg<BM, BN>;
    using L = OperandLayout<LAYOUT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);

    const int S = p.stages;
    uint8_t *smA = smem;
    uint8_t *smB = smem + S * Cfg::A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smB + S * Cfg::B_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + S;
    uint64_t *acc_full = bars + 2 * S;       // [2]
    uint64_t *acc_empty = bars + 2 * S + 2;  // [2]
    uint64_t *mma_done = bars + 2 * S + 4;
    volatile uint32_t *ctrl = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 5);
    // ctrl[0]: TMEM base   ctrl[1]: error flag   ctrl[2]: k-tiles issued by TMA

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long nK = p.num_k_tiles;
    const long long U = static_cast<long long>(p.num_m_tiles) * p.num_n_tiles * nK;
    const long long G = gridDim.x;
    const long long u_begin = sk_first_unit(blockIdx.x, G, U);
    const long long u_end = sk_first_unit(static_cast<long long>(blockIdx.x) + 1, G, U);
    const uint64_t lim = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), Cfg::EPI_WARPS);
        }
        mbar_init(smem_u32(mma_done), 1);
        ctrl[1] = 0;
        ctrl[2] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(&ctrl[0])), Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctrl[0];
    griddep_launch_dependents();
    griddep_wait();  // the previous kernel's writes (A, B, C, counters) are visible from here on

    // Segments of this CTA: (tile, k-tiles [kb, ke)); every role walks the same list
    // with `for (long long u_ = u_begin; u_ < u_end;) { const SkSegment sg = sk_next(...)`.

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int s = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool stop = false;
            // per-slot addresses are fixed offsets from slot 0 (see gemm_kernel.cuh)
            const uint32_t empty0 = smem_u32(&empty[0]), full0 = smem_u32(&full[0]);
            const uint32_t smA0 = smem_u32(smA), smB0 = smem_u32(smB);
            for (long long u_ = u_begin; u_ < u_end;) {
                const SkSegment sg_ = sk_next(u_, u_end, nK);
                const int tile = sg_.tile, kb = sg_.kb, ke = sg_.ke;
                if (stop) break;
                int m_tile, n_tile;
                tile_coords(tile, p.num_m_tiles, p.num_n_tiles, p.raster_group, m_tile, n_tile);
                const int m0 = m_tile * BM, n0 = n_tile * BN;
// (the k-loops of the producer and MMA threads are unrolled by four: these single
// threads set the pace of a k-tile, and the unrolled loop issues fewer instructions)
#pragma unroll 4
                for (int kt = kb; kt < ke; ++kt) {
                    if (!mbar_wait_for(empty0 + 8u * s, phase ^ 1u, lim)) {
                        record_status(p.status, kSiteProducer);
                        ctrl[1] = 1;
                        stop = true;
                        break;
                    }
                    if ((kt & 7) == 0 && ctrl[1]) { stop = true; break; }
                    const uint32_t fb = full0 + 8u * s;
                    mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    load_operand<false, L::A_MN, BM, BM>(smA0 + static_cast<uint32_t>(s) * Cfg::A_BYTES, &tmA, fb, kt,
                                                         m0);
                    load_operand<false, L::B_MN, BN, (BN < 64 ? BN : 64)>(smB0 + static_cast<uint32_t>(s) * Cfg::B_BYTES,
                                                                         &tmB, fb, kt, n0);
                    ++issued;
                    if (++s == S) { s = 0; phase ^= 1u; }
                }
            }
            ctrl[2] = issued;  // read by the drain after an error, once every role has stopped
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            const uint32_t idesc = idesc_for(p.idesc_flags, BM, BN);
            constexpr uint64_t a_step = operand_k_step<L::A_MN>(), b_step = operand_k_step<L::B_MN>();
            int s = 0;
            uint32_t phase = 0;
            int j = 0;
            bool stop = false;
            const uint64_t a_desc0 = operand_desc<L::A_MN>(smem_u32(smA));
            const uint64_t b_desc0 = operand_desc<L::B_MN>(smem_u32(smB));
            const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
            for (long long u_ = u_begin; u_ < u_end;) {
                const SkSegment sg_ = sk_next(u_, u_end, nK);
                const int tile = sg_.tile, kb = sg_.kb, ke = sg_.ke;
                if (stop) break;
                (void)tile;
                const int b = j & 1;
                const uint32_t acc_phase = static_cast<uint32_t>((j >> 1) & 1);
                ++j;
                if (!mbar_wait_for(smem_u32(&acc_empty[b]), acc_phase ^ 1u, lim)) {
                    record_status(p.status, kSiteMma);
                    ctrl[1] = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll 4
                for (int kt = kb; kt < ke; ++kt) {
                    if (!mbar_wait_for(full0 + 8u * s, phase, lim)) {
                        record_status(p.status, kSiteMma);
                        ctrl[1] = 1;
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(s) * (Cfg::A_BYTES >> 4);
                    const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(s) * (Cfg::B_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma_f16(d_tmem, a_desc + a_step * kk, b_desc + b_step * kk, idesc,
                                 (kt > kb || kk > 0) ? 1u : 0u);
                    umma_commit(empty0 + 8u * s);
                    if (++s == S) { s = 0; phase ^= 1u; }
                }
                if (!stop) umma_commit(smem_u32(&acc_full[b]));
            }
            // all MMAs this thread issued have completed once mma_done flips
            umma_commit(smem_u32(mma_done));
            if (!mbar_wait_for(smem_u32(mma_done), 0, lim)) record_status(p.status, kSiteDrain);
        }
    } else {
        // ---------------- epilogue warps ----------------
        const int q = warp & 3;
        // Accumulator row r sits in TMEM lane r for M = 128; for M = 64 rows
        // 16q .. 16q+15 sit in lanes 32q .. 32q+15 of lane quarter q.
        const int r = (BM == 128) ? (q * 32 + lane) : (q * 16 + lane);
        const bool lane_has_row = (BM == 128) || (lane < 16);
        const bool bf16 = ((p.idesc_flags >> 7) & 7u) == 1u;
        constexpr int CH = BN < 32 ? BN : 32;  // accumulator columns per TMEM load
        int j = 0;
        for (long long u_ = u_begin; u_ < u_end;) {
                const SkSegment sg_ = sk_next(u_, u_end, nK);
                const int tile = sg_.tile, kb = sg_.kb, ke = sg_.ke;
            const int b = j & 1;
            const uint32_t acc_phase = static_cast<uint32_t>((j >> 1) & 1);
            const int slot = 2 * static_cast<int>(blockIdx.x) + (j == 0 ? 0 : 1);
            ++j;
            if (!warp_wait(smem_u32(&acc_full[b]), acc_phase, 4 * lim, lane)) {
                if (lane == 0) {
                    record_status(p.status, kSiteEpilogue);
                    ctrl[1] = 1;
                }
                break;
            }
            tc_fence_after();
            int m_tile, n_tile;
            tile_coords(tile, p.num_m_tiles, p.num_n_tiles, p.raster_group, m_tile, n_tile);
            const int m0 = m_tile * BM, n0 = n_tile * BN;
            const bool whole = (kb == 0 && ke == nK);
            const bool row_ok = lane_has_row && (m0 + r < p.M);
            const uint32_t taddr = tmem_base + static_cast<uint32_t>(b * BN) + (static_cast<uint32_t>(q * 32) << 16);
            float *prow = p.partials + (static_cast<size_t>(slot) * BM + r) * BN;
#pragma unroll 1
            for (int c = 0; c < BN; c += CH) {
                uint32_t v[32];
                if (CH == 32) tmem_ld_32x32b_x32(taddr + c, v);
                else tmem_ld_32x32b_x16(taddr + c, v);
                tmem_ld_wait();
                if (c + CH == BN) {
                    // the whole accumulator of this segment is in registers: hand the buffer back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
                }
                if (!row_ok) continue;
#pragma unroll
                for (int t = 0; t < CH; t += 8) {
                    const float4 lo = make_float4(__uint_as_float(v[t]), __uint_as_float(v[t + 1]),
                                                  __uint_as_float(v[t + 2]), __uint_as_float(v[t + 3]));
                    const float4 hi = make_float4(__uint_as_float(v[t + 4]), __uint_as_float(v[t + 5]),
                                                  __uint_as_float(v[t + 6]), __uint_as_float(v[t + 7]));
                    if (whole) {
                        sk_store8(p, m0 + r, n0 + c + t, lo, hi, bf16);
                    } else {
                        reinterpret_cast<float4 *>(prow + c + t)[0] = lo;
                        reinterpret_cast<float4 *>(prow + c + t)[1] = hi;
                    }
                }
            }
            // A quarter with no row inside C takes no part in the fix-up (every CTA of
            // the tile skips it alike, so its counter stays untouched).
            const int row0 = BM == 128 ? q * 32 : q * 16;
            if (!whole && m0 + row0 < p.M && p.splitk_reduce_in_kernel) {
                // Publish this quarter's partial rows, then count the arrival on the
                // (tile, quarter) counter; the last of the tile's CTAs to arrive sums.
                __threadfence();
                __syncwarp();
                const long long u0 = static_cast<long long>(tile) * nK;
                const int g_lo = sk_owner(u0, G, U), g_hi = sk_owner(u0 + nK - 1, G, U);
                unsigned last = 0;
                if (lane == 0) {
                    const unsigned prev = atomicAdd(&p.counters[static_cast<size_t>(tile) * 4 + q], 1u);
                    last = (prev + 1 == static_cast<unsigned>(g_hi - g_lo + 1)) ? 1u : 0u;
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    // The quarter's rows (32, or 16 for BM = 64) x BN columns, 256 elements
                    // per step: lane l takes 8 consecutive columns, so each load of the
                    // warp reads whole 32-byte sectors of a slot row and each store
                    // writes 16 bytes of a C row.  Partial rows beyond M were never
                    // written and are not stored.
                    constexpr int R = BM == 128 ? 32 : 16;
                    static_assert((R * BN) % 1024 == 0 || R * BN == 256 || R * BN == 512, "whole steps");
                    const int vrows = min(R, p.M - m0 - row0);      // rows of the quarter inside C
                    const int steps = (vrows * BN + 255) / 256;      // 256 elements per step
                    // slot of CTA g for this tile: 2g when the tile is g's first, else 2g+1
                    const int lo_slot = 2 * g_lo + (sk_first_unit(g_lo, G, U) / nK == tile ? 0 : 1);
                    // Up to four steps at a time: for each CTA in order, all of its loads of
                    // those steps are issued before any is used; the sum starts from the
                    // first CTA's partial and adds the others in CTA order.
#pragma unroll 1
                    for (int st0 = 0; st0 < steps; st0 += 4) {
                        float4 acc[8];
#pragma unroll 2
                        for (int g = g_lo; g <= g_hi; ++g) {
                            const int sl = g == g_lo ? lo_slot : 2 * g;
                            const float *slot_base = p.partials + static_cast<size_t>(sl) * BM * BN;
                            float4 x[8];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int e = (st0 + i) * 256 + lane * 8;
                                const float *src = slot_base + static_cast<size_t>(row0) * BN + e;
                                if (st0 + i < steps) {
                                    x[2 * i] = __ldcg(reinterpret_cast<const float4 *>(src));
                                    x[2 * i + 1] = __ldcg(reinterpret_cast<const float4 *>(src + 4));
                                } else {
                                    x[2 * i] = x[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                                }
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                if (g == g_lo) {
                                    acc[i] = x[i];
                                } else {
                                    acc[i].x += x[i].x; acc[i].y += x[i].y; acc[i].z += x[i].z; acc[i].w += x[i].w;
                                }
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int e = (st0 + i) * 256 + lane * 8;
                            const int rr = row0 + e / BN, cc = e % BN;
                            if (st0 + i < steps && rr - row0 < vrows) sk_store8(p, m0 + rr, n0 + cc, acc[2 * i], acc[2 * i + 1], bf16);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) p.counters[static_cast<size_t>(tile) * 4 + q] = 0u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && ctrl[1]) {
        const int issued = static_cast<int>(ctrl[2]);
        for (int i = max(0, issued - S); i < issued; ++i) {
            if (!mbar_wait_for(smem_u32(&full[i % S]), static_cast<uint32_t>((i / S) & 1), lim)) {
                record_status(p.status, kSiteDrain);
                break;
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BM, int BN, int LAYOUT>
int launch_gemm_streamk(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &args,
                        cudaStream_t stream);

}  // namespace sdt
