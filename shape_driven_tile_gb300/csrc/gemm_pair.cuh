// gemm_pair.cuh -- persistent two-CTA (cta_group::2) tcgen05 fp16 GEMM.
//
// A cluster of two CTAs on neighbouring SMs computes one 256 x BN output tile
// with a single stream of M=256 MMAs issued by the leader CTA (cluster rank 0):
//   - each CTA stages, per k-tile, its own 128 rows of A and its own BN/2
//     columns of B (same smem offsets in both CTAs); the MMA reads A rows and B
//     columns from both SMs, so every operand byte is fetched from L2 once per
//     pair instead of once per CTA -- a 256 x BN pair moves (128 + BN/2) x 64 x 2
//     bytes per SM per k-tile against (128 + BN) x 64 x 2 for a 128 x BN CTA;
//   - the accumulator of rows 0-127 lives in the leader's TMEM, rows 128-255 in
//     the peer's, each 128 lanes x BN columns, double-buffered as in
//     gemm_persistent.cuh;
//   - both CTAs' TMA loads complete on the leader's "full" barrier (armed by the
//     leader with both CTAs' bytes); the leader's commits arrive on the "empty"
//     and "acc_full" barriers of both CTAs (multicast); both CTAs' epilogue warps
//     arrive on the leader's "acc_empty" barrier.
// Everything else (tile walk, ring, epilogue, bounded waits) follows
// gemm_persistent.cuh.
#pragma once

#include <cuda_fp16.h>

#include "gemm_kernel.cuh"
#include "gemm_persistent.cuh"
#include "ptx.cuh"

namespace sdt {

template <int BN>
struct PairCfg {
    static constexpr int BM = 256;     // rows per pair tile
    static constexpr int CTA_M = 128;  // rows staged and accumulated per CTA
    static constexpr int B_HALF = BN / 2;  // B columns each CTA stages and supplies to the MMA
    // MN-major B arrives in whole 64-column boxes (BN = 224: two boxes for 112 columns);
    // K-major B in one box of B_HALF rows when B_HALF is not a multiple of 64
    static constexpr int B_SMEM_COLS = (B_HALF + 63) / 64 * 64;
    static constexpr int B_KBOX = B_HALF % 64 == 0 ? 64 : B_HALF;
    static constexpr int A_BYTES = CTA_M * kBK * 2;
    static constexpr int B_BYTES = B_SMEM_COLS * kBK * 2;  // shared memory per stage
    static constexpr int B_BOX_BYTES = 64 * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // per CTA
    static constexpr int ACC_BUFS = 2;
    // two accumulators of BN columns; the allocation is a power of two
    static constexpr int TMEM_COLS = ACC_BUFS * BN <= 256 ? 256 : 512;
    // bytes one CTA's TMA copies bring per k-tile (whole tile; B as it is staged)
    template <bool B_MN>
    __host__ __device__ static constexpr int load_bytes() {
        return A_BYTES + (B_MN ? B_SMEM_COLS : B_HALF) * kBK * 2;
    }
    static constexpr int THREADS = 192;
    static constexpr int EPI_WARPS = 4;
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int CTRL_BYTES = 512;
    static constexpr int C_STAGE_BYTES = EPI_WARPS * 2 * kCStageBytes;  // C staging, two buffers per epilogue warp
    __host__ __device__ static constexpr int smem_bytes(int stages) {
        return ALIGN_SLACK + stages * STAGE_BYTES + C_STAGE_BYTES + CTRL_BYTES;
    }
    static_assert(BN == 128 || BN == 224 || BN == 256, "pair tiles use BN 128, 224 or 256");
    static_assert(ACC_BUFS * BN <= TMEM_COLS && TMEM_COLS <= 512, "two accumulators must fit in TMEM");
};

// Work item -> output tile, column offset and width.  When the last round of whole
// tiles would leave at least half of the pairs idle, the host makes each of those
// tail tiles two half-width items instead, so the tail takes half a round.
template <int BN>
__device__ __forceinline__ void pair_item(int item, const GemmArgs &p, int &tile, int &m_tile, int &n_tile,
                                          int &n_off, int &width) {
    if (item < p.tail_start) {
        tile = item;
        n_off = 0;
        width = BN;
    } else {
        const int h = item - p.tail_start;
        tile = p.tail_start + (h >> 1);
        n_off = (h & 1) * (BN / 2);
        width = BN / 2;
    }
    tile_coords(tile, p.num_m_tiles, p.num_n_tiles, p.raster_group, m_tile, n_tile);
}

template <int BN, int LAYOUT>
__global__ void __launch_bounds__(192, 1)
    gemm_f16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const GemmArgs p) {
    using Cfg = PairCfg<BN>;
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
    uint64_t *acc_full = bars + 2 * S;
    uint64_t *acc_empty = bars + 2 * S + 2;
    uint64_t *mma_done = bars + 2 * S + 4;
    volatile uint32_t *ctrl = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 5);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int num_pairs = static_cast<int>(gridDim.x >> 1);
    const int num_items = p.num_items;  // whole tiles (256 rows each) and tail halves
    const int nK = p.num_k_tiles;
    const uint64_t lim = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 2 * Cfg::EPI_WARPS);
        }
        mbar_init(smem_u32(mma_done), 1);
        ctrl[1] = 0;
        ctrl[2] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(&ctrl[0])), Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both SMs
    tc_fence_after();
    const uint32_t tmem_base = ctrl[0];
    griddep_wait();  // the previous kernel's writes (A, B, C) are visible from here on

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int s = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool stop = false;
            // per-slot addresses are fixed offsets from slot 0 (the leader's full barrier
            // keeps its offset under mapa), so the loop adds instead of recomputing them
            const uint32_t empty0 = smem_u32(&empty[0]), full0 = smem_u32(&full[0]);
            const uint32_t full0_leader = mapa_shared(full0, 0);
            const uint32_t smA0 = smem_u32(smA), smB0 = smem_u32(smB);
            for (int item = pair; item < num_items && !stop; item += num_pairs) {
                int tile, m_tile, n_tile, n_off, width;
                pair_item<BN>(item, p, tile, m_tile, n_tile, n_off, width);
                const int m0 = m_tile * Cfg::BM + static_cast<int>(rank) * Cfg::CTA_M;
                const int nb = n_tile * BN + n_off + static_cast<int>(rank) * (width / 2);
                const bool whole = width == BN;  // whole tile, else a tail half (BN/4 B rows per CTA)
                // the next kernel in the stream may be launched once every CTA starts its
                // last item: a dependent that fits beside this kernel (a decode GEMV) then
                // prefetches near the end of this launch instead of at its start
                if (item + num_pairs >= num_items) griddep_launch_dependents();
                const uint32_t pair_bytes = 2u * static_cast<uint32_t>(
                    whole ? Cfg::template load_bytes<L::B_MN>() : Cfg::A_BYTES + (Cfg::B_HALF / 2) * kBK * 2);
                const int start =
                    p.stagger ? static_cast<int>((static_cast<uint32_t>(tile) * static_cast<uint32_t>(p.stagger_stride)) &
                                                 static_cast<uint32_t>(nK - 1))
                              : 0;
// (the k-loops of the producer and MMA threads are unrolled by four: these single
// threads set the pace of a k-tile, and the unrolled loop issues fewer instructions)
#pragma unroll 4
                for (int i = 0; i < nK; ++i) {
                    if (!mbar_wait_for(empty0 + 8u * s, phase ^ 1u, lim)) {
                        record_status(p.status, kSiteProducer | static_cast<int>(rank << 4) | (issued << 8));
                        ctrl[1] = 1;
                        stop = true;
                        break;
                    }
                    if ((i & 7) == 0 && ctrl[1]) { stop = true; break; }  // another role gave up
                    const int kt = p.stagger ? ((start + i) & (nK - 1)) : i;
                    if (leader) mbar_arrive_expect_tx(full0 + 8u * s, pair_bytes);
                    const uint32_t fb = full0_leader + 8u * s;
                    const uint32_t dA = smA0 + static_cast<uint32_t>(s) * Cfg::A_BYTES;
                    const uint32_t dB = smB0 + static_cast<uint32_t>(s) * Cfg::B_BYTES;
                    load_operand<true, L::A_MN, Cfg::CTA_M, Cfg::CTA_M>(dA, &tmA, fb, kt, m0);
                    if constexpr (Cfg::B_HALF == 128) {
                        if (whole)
                            load_operand<true, L::B_MN, Cfg::B_HALF, 64>(dB, &tmB, fb, kt, nb);
                        else
                            load_operand<true, L::B_MN, Cfg::B_HALF / 2, 64>(dB, &tmB, fb, kt, nb);
                    } else {  // tail halves only for BN = 256 (the host splits no other tail)
                        load_operand<true, L::B_MN, Cfg::B_HALF, Cfg::B_KBOX>(dB, &tmB, fb, kt, nb);
                    }
                    ++issued;
                    if (++s == S) { s = 0; phase ^= 1u; }
                }
            }
            ctrl[2] = issued;  // read by the drain after an error, once every role has stopped
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader only) ----------------
            const uint32_t idesc_full = idesc_for(p.idesc_flags, Cfg::BM, BN);
            const uint32_t idesc_half = idesc_for(p.idesc_flags, Cfg::BM, BN / 2);
            constexpr uint64_t a_step = operand_k_step<L::A_MN>(), b_step = operand_k_step<L::B_MN>();
            int s = 0;
            uint32_t phase = 0;
            int j = 0;
            bool stop = false;
            // slot s's descriptors are slot 0's plus s stages (the start address field
            // counts 16-byte units and shared memory stays below 2^18 bytes)
            const uint64_t a_desc0 = operand_desc<L::A_MN>(smem_u32(smA));
            const uint64_t b_desc0 = operand_desc<L::B_MN>(smem_u32(smB));
            const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
            for (int item = pair; item < num_items && !stop; item += num_pairs, ++j) {
                const uint32_t idesc = item < p.tail_start ? idesc_full : idesc_half;
                const int b = j & 1;
                const uint32_t acc_phase = static_cast<uint32_t>((j >> 1) & 1);
                if (!mbar_wait_cluster_for(smem_u32(&acc_empty[b]), acc_phase ^ 1u, lim)) {
                    record_status(p.status, kSiteMma | 0x80 | (j << 8));
                    ctrl[1] = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll 4
                for (int i = 0; i < nK; ++i) {
                    if (!mbar_wait_for(full0 + 8u * s, phase, lim)) {
                        record_status(p.status, kSiteMma | (((j << 12) | i) << 8));
                        ctrl[1] = 1;
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(s) * (Cfg::A_BYTES >> 4);
                    const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(s) * (Cfg::B_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma_f16_pair(d_tmem, a_desc + a_step * kk, b_desc + b_step * kk, idesc,
                                      (i > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_pair(empty0 + 8u * s, 0x3);
                    if (++s == S) { s = 0; phase ^= 1u; }
                }
                if (!stop) umma_commit_pair(smem_u32(&acc_full[b]), 0x3);
            }
            umma_commit_pair(smem_u32(mma_done), 0x1);
            if (!mbar_wait_for(smem_u32(mma_done), 0, lim)) record_status(p.status, kSiteDrain);
        }
    } else {
        // ---------------- epilogue warps (both CTAs) ----------------
        const int q = warp & 3;
        const uint32_t cbuf = smem_u32(smC) + static_cast<uint32_t>(q) * 2u * kCStageBytes;
        int nst = 0;  // TMA stores this warp has issued (staging buffer parity)
        int j = 0;
        for (int item = pair; item < num_items; item += num_pairs, ++j) {
            const int b = j & 1;
            const uint32_t acc_phase = static_cast<uint32_t>((j >> 1) & 1);
            if (!warp_wait(smem_u32(&acc_full[b]), acc_phase, 4 * lim, lane)) {
                if (lane == 0) {
                    record_status(p.status, kSiteEpilogue | static_cast<int>(rank << 4) | (j << 8));
                    ctrl[1] = 1;
                }
                break;
            }
            tc_fence_after();
            int tile, m_tile, n_tile, n_off, width;
            pair_item<BN>(item, p, tile, m_tile, n_tile, n_off, width);
            const int row0 = m_tile * Cfg::BM + static_cast<int>(rank) * Cfg::CTA_M + q * 32;  // this warp's rows
            const int n0 = n_tile * BN + n_off;
            const bool bf16 = ((p.idesc_flags >> 7) & 7u) == 1u;
            const uint32_t taddr =
                tmem_base + static_cast<uint32_t>(b * BN) + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < width; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c, r);
                tmem_ld_wait();
                if (c == width - 32) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[b]), 0));
                }
                store_chunk_tma(&tmC, cbuf, nst++, r, bf16, n0 + c, row0, lane);
            }
        }
        if (lane == 0) bulk_wait_group<0>();  // this warp's stores have landed (and read the staging)
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && leader && ctrl[1]) {
        const int issued = static_cast<int>(ctrl[2]);
        for (int i = max(0, issued - S); i < issued; ++i) {
            if (!mbar_wait_for(smem_u32(&full[i % S]), static_cast<uint32_t>((i / S) & 1), lim)) {
                record_status(p.status, kSiteDrain);
                break;
            }
        }
    }
    cluster_sync();  // both CTAs done with each other's smem, barriers and TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN, int LAYOUT>
int launch_gemm_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &args,
                     cudaStream_t stream);

}  // namespace sdt
