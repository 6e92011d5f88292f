// gemm_persistent.cuh -- persistent, warp-specialised tcgen05 fp16 GEMM with a
// double-buffered TMEM accumulator (one CTA per SM, BM = 128).
//
// Same arithmetic as gemm_kernel.cuh (fp16 operands, fp32 accumulation in
// tensor memory, fp16 output) and the same TMA/descriptor layouts; what changes
// is the schedule.  The grid is at most one CTA per SM and each CTA walks the
// output tiles b, b + gridDim.x, b + 2*gridDim.x, ... (banded raster order), so
//   - the smem ring keeps streaming across tile boundaries (no pipeline refill),
//   - the accumulator alternates between two TMEM buffers: while the epilogue
//     warps drain tile j from buffer j%2, the MMA warp already accumulates tile
//     j+1 into the other buffer.
//
// Roles (192 threads):
//   warp 0 lane 0 : TMA producer (ring slots: full/empty mbarriers)
//   warp 1        : TMEM allocation; lane 0 issues tcgen05.mma and commits
//   warps 2..5    : epilogue; warp w reads TMEM lane quarter w % 4
// Accumulator hand-off: acc_full[b] (MMA commit -> epilogue) and acc_empty[b]
// (one arrival per epilogue warp -> MMA).
//
// Every wait is bounded per wait (p.timeout_ns from the first failed poll); on
// expiry the kernel records the site in the status word and unwinds: the
// producer stops issuing, the MMA warp waits for its own MMAs, outstanding TMA
// copies are drained, TMEM is freed.
#pragma once

#include <cuda_fp16.h>

#include "gemm_kernel.cuh"
#include "ptx.cuh"

namespace sdt {

template <int BN>
struct PersistentCfg {
    static constexpr int BM = 128;
    static constexpr int A_BYTES = BM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int B_BOX_BYTES = 64 * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = ACC_BUFS * BN;
    static constexpr int THREADS = 192;
    static constexpr int EPI_WARPS = 4;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int CTRL_BYTES = 512;
    static constexpr int C_STAGE_BYTES = EPI_WARPS * 2 * kCStageBytes;  // C staging, two buffers per epilogue warp
    __host__ __device__ static constexpr int smem_bytes(int stages) {
        return ALIGN_SLACK + stages * STAGE_BYTES + C_STAGE_BYTES + CTRL_BYTES;
    }
    static_assert(BN == 128 || BN == 256, "persistent tiles use BN 128 or 256");
    static_assert(TMEM_COLS <= 512, "two accumulators must fit in TMEM");
};

// Banded raster: tile index -> (m_tile, n_tile); bands of `group` m-tiles, m fastest.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group, int &m_tile,
                                            int &n_tile) {
    const int per_band = group * num_n;
    const int band = tile / per_band;
    const int first_m = band * group;
    const int band_m = min(num_m - first_m, group);
    const int in_band = tile - band * per_band;
    m_tile = first_m + in_band % band_m;
    n_tile = in_band / band_m;
}

template <int BN, int LAYOUT>
__global__ void __launch_bounds__(192, 1)
    gemm_f16_persistent_kernel(const __grid_constant__ CUtensorMap tmA,
                               const __grid_constant__ CUtensorMap tmB,
                               const __grid_constant__ CUtensorMap tmC, const GemmArgs p) {
    using Cfg = PersistentCfg<BN>;
    using L = OperandLayout<LAYOUT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);

    const int S = p.stages;
    uint8_t *smA = smem;
    uint8_t *smB = smem + S * Cfg::A_BYTES;
    uint8_t *smC = smB + S * Cfg::B_BYTES;  // C staging (1024-byte aligned)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smC + Cfg::C_STAGE_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + S;
    uint64_t *acc_full = bars + 2 * S;       // [2]
    uint64_t *acc_empty = bars + 2 * S + 2;  // [2]
    uint64_t *mma_done = bars + 2 * S + 4;
    volatile uint32_t *ctrl = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 5);
    // ctrl[0]: TMEM base   ctrl[1]: error flag   ctrl[2]: k-tiles issued by TMA

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = p.num_m_tiles * p.num_n_tiles;
    const int nK = p.num_k_tiles;
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
    griddep_wait();  // the previous kernel's writes (A, B, C) are visible from here on

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int s = 0;
            uint32_t phase = 0;
            int issued = 0;
            // per-slot addresses are fixed offsets from slot 0 (see gemm_kernel.cuh)
            const uint32_t empty0 = smem_u32(&empty[0]), full0 = smem_u32(&full[0]);
            const uint32_t smA0 = smem_u32(smA), smB0 = smem_u32(smB);
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                // dependents may launch once every CTA starts its last tile (see gemm_pair.cuh)
                if (tile + static_cast<int>(gridDim.x) >= num_tiles) griddep_launch_dependents();
                int m_tile, n_tile;
                tile_coords(tile, p.num_m_tiles, p.num_n_tiles, p.raster_group, m_tile, n_tile);
                const int m0 = m_tile * Cfg::BM, n0 = n_tile * BN;
                const int start =
                    p.stagger ? static_cast<int>((static_cast<uint32_t>(tile) * static_cast<uint32_t>(p.stagger_stride)) &
                                                 static_cast<uint32_t>(nK - 1))
                              : 0;
                bool stop = false;
// (the k-loops of the producer and MMA threads are unrolled by four: these single
// threads set the pace of a k-tile, and the unrolled loop issues fewer instructions)
#pragma unroll 4
                for (int i = 0; i < nK; ++i) {
                    if (!mbar_wait_for(empty0 + 8u * s, phase ^ 1u, lim)) {
                        record_status(p.status, kSiteProducer);
                        ctrl[1] = 1;
                        stop = true;
                        break;
                    }
                    if ((i & 7) == 0 && ctrl[1]) { stop = true; break; }
                    const int kt = p.stagger ? ((start + i) & (nK - 1)) : i;
                    const uint32_t fb = full0 + 8u * s;
                    mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    load_operand<false, L::A_MN, Cfg::BM, Cfg::BM>(smA0 + static_cast<uint32_t>(s) * Cfg::A_BYTES, &tmA,
                                                                   fb, kt, m0);
                    load_operand<false, L::B_MN, BN, 64>(smB0 + static_cast<uint32_t>(s) * Cfg::B_BYTES, &tmB, fb, kt,
                                                         n0);
                    ++issued;
                    if (++s == S) { s = 0; phase ^= 1u; }
                }
                if (stop) break;
            }
            ctrl[2] = issued;  // read by the drain after an error, once every role has stopped
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            const uint32_t idesc = idesc_for(p.idesc_flags, Cfg::BM, BN);
            constexpr uint64_t a_step = operand_k_step<L::A_MN>(), b_step = operand_k_step<L::B_MN>();
            int s = 0;
            uint32_t phase = 0;
            int j = 0;
            bool stop = false;
            const uint64_t a_desc0 = operand_desc<L::A_MN>(smem_u32(smA));
            const uint64_t b_desc0 = operand_desc<L::B_MN>(smem_u32(smB));
            const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
            for (int tile = blockIdx.x; tile < num_tiles && !stop; tile += gridDim.x, ++j) {
                const int b = j & 1;
                const uint32_t acc_phase = static_cast<uint32_t>((j >> 1) & 1);
                if (!mbar_wait_for(smem_u32(&acc_empty[b]), acc_phase ^ 1u, lim)) {
                    record_status(p.status, kSiteMma);
                    ctrl[1] = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll 4
                for (int i = 0; i < nK; ++i) {
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
                                 (i > 0 || kk > 0) ? 1u : 0u);
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
        const uint32_t cbuf = smem_u32(smC) + static_cast<uint32_t>(q) * 2u * kCStageBytes;
        int nst = 0;  // TMA stores this warp has issued (staging buffer parity)
        int j = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++j) {
            const int b = j & 1;
            const uint32_t acc_phase = static_cast<uint32_t>((j >> 1) & 1);
            if (!warp_wait(smem_u32(&acc_full[b]), acc_phase, lim, lane)) {
                if (lane == 0) {
                    record_status(p.status, kSiteEpilogue);
                    ctrl[1] = 1;
                }
                break;
            }
            tc_fence_after();
            int m_tile, n_tile;
            tile_coords(tile, p.num_m_tiles, p.num_n_tiles, p.raster_group, m_tile, n_tile);
            const int row0 = m_tile * Cfg::BM + q * 32;  // this warp's rows
            const int n0 = n_tile * BN;
            const bool bf16 = ((p.idesc_flags >> 7) & 7u) == 1u;
            const uint32_t taddr = tmem_base + static_cast<uint32_t>(b * BN) + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c, r);
                tmem_ld_wait();
                if (c == BN - 32) {
                    // the whole accumulator of this tile is in registers: hand the buffer back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
                }
                store_chunk_tma(&tmC, cbuf, nst++, r, bf16, n0 + c, row0, lane);
            }
        }
        if (lane == 0) bulk_wait_group<0>();  // this warp's stores have landed (and read the staging)
        __syncwarp();
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

template <int BN, int LAYOUT>
int launch_gemm_persistent(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                           const GemmArgs &args, cudaStream_t stream);

}  // namespace sdt
