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
//
// The last round of a launch whose tiles do not fill every pair runs in one of two
// forms, both planned on the host: each leftover tile as two half-width items, or,
// given a workspace, each leftover tile as S full-width items over consecutive
// k-ranges whose fp32 partials are summed by the last of them to finish (below).
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

// Work item -> output tile, column offset, width and k-range.  Items [0, tail_start)
// are whole tiles over all k-tiles.  The items after them cover the tiles left for a
// last, partly empty round: with p.tail_splits == 0 two half-width items per tile;
// with p.tail_splits = S >= 2, S full-width items per tile over consecutive k-ranges
// (split >= 0 marks such an item): split 0 takes the first p.tail_long k-tiles and
// the other S-1 share the rest evenly (p.tail_long == 0: all S share nK evenly).
// A longer split 0 is meant to finish last, after the others' partials are out.
template <int BN, bool KSPLIT>
__device__ __forceinline__ void pair_item(int item, const GemmArgs &p, int &tile, int &m_tile, int &n_tile,
                                          int &n_off, int &width, int &k0, int &kn, int &split) {
    const int nK = p.num_k_tiles;
    n_off = 0;
    width = BN;
    k0 = 0;
    kn = nK;
    split = -1;
    if (item < p.tail_start) {
        tile = item;
    } else if (KSPLIT) {
        const int h = item - p.tail_start;
        split = h % p.tail_splits;
        tile = p.tail_start + h / p.tail_splits;
        if (p.tail_long <= 0) {
            k0 = split * nK / p.tail_splits;
            kn = (split + 1) * nK / p.tail_splits - k0;
        } else if (split == 0) {
            kn = p.tail_long;
        } else {
            const int rest = nK - p.tail_long, others = p.tail_splits - 1;
            k0 = p.tail_long + (split - 1) * rest / others;
            kn = p.tail_long + split * rest / others - k0;
        }
    } else {
        const int h = item - p.tail_start;
        tile = p.tail_start + (h >> 1);
        n_off = (h & 1) * (BN / 2);
        width = BN / 2;
    }
    tile_coords(tile, p.num_m_tiles, p.num_n_tiles, p.raster_group, m_tile, n_tile);
}

// Copy buffers (and mbarriers) per epilogue warp for a k-split tail's partials (S >= 3),
// and the 32-column chunks of the other partial a warp keeps in flight when S == 2.
constexpr int kTailBufs = 4;
constexpr int kTailAhead = 2;

// Warp-uniform bounded wait for an mbarrier phase that also watches a u32 counter in
// global memory: 1 once the phase has completed (every lane then observes it), 2 as
// soon as lane 0 reads `want` from the counter first (acquire; the phase may still be
// pending), 0 when `limit_ns` passes.
__device__ __forceinline__ int warp_wait_or_count(uint32_t bar, uint32_t parity, const unsigned *ctr, unsigned want,
                                                  uint64_t limit_ns, int lane) {
    int st = 0;
    if (lane == 0) {
        if (mbar_try_wait(bar, parity)) {
            st = 1;
        } else {
            const uint64_t deadline = global_timer_ns() + limit_ns;
            for (uint32_t polls = 1;; ++polls) {
                if (mbar_try_wait(bar, parity)) { st = 1; break; }
                if ((polls & 7u) == 0) {
                    unsigned seen;
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(ctr) : "memory");
                    if (seen == want) { st = 2; break; }
                    if (global_timer_ns() > deadline) break;
                }
                __nanosleep(32);
            }
        }
    }
    st = __shfl_sync(0xffffffffu, st, 0);
    if (st == 1 && lane != 0 && !mbar_wait_for(bar, parity, limit_ns)) st = 0;
    return __all_sync(0xffffffffu, st != 0) ? st : 0;
}

// The (tile, CTA, epilogue warp) arrival counter of k-split tail item h.
__device__ __forceinline__ unsigned *pair_tail_counter(const GemmArgs &p, int h, uint32_t rank, int q) {
    return p.counters + (static_cast<size_t>(h / p.tail_splits) * 2 + rank) * 4 + static_cast<size_t>(q);
}

// Workspace slot of a k-split tail item's partial: item h = item - tail_start, this CTA
// (rank) and epilogue warp q own 32 rows x BN fp32 values.  Within the slot, columns
// [c, c+32) of lane l (row l of the warp's 32) are the eight float4 at float offsets
// c*32 + j*128 + l*4, j = 0..7: a warp's 16-byte stores and loads each cover 512
// contiguous bytes, and any run of whole 32-column chunks is one contiguous range.
template <int BN>
__device__ __forceinline__ float *pair_tail_slot(const GemmArgs &p, int h, uint32_t rank, int q) {
    return p.partials + ((static_cast<size_t>(h) * 2 + rank) * 4 + static_cast<size_t>(q)) * (32 * BN);
}

// The first `chunks` (at most kTailAhead) 32-column chunks of a partial, lane's row.
__device__ __forceinline__ void pair_tail_load_ahead(const float4 *oth, int chunks, float4 (&ahead)[kTailAhead][8]) {
#pragma unroll
    for (int d = 0; d < kTailAhead; ++d)
        if (d < chunks) {
#pragma unroll
            for (int j = 0; j < 8; ++j) ahead[d][j] = __ldcg(oth + d * 256 + 32 * j);
        }
}

// Epilogue of one k-split tail item, for one warp's 32 rows (lane = row).  A warp
// that finds the (tile, rank, warp) counter at S-1 -- every other split has already
// published its partial -- is the last and skips publishing its own.  Otherwise it
// writes its partial to its slot and then counts its arrival; the one whose count
// makes S is the last.  The last warp -- whichever split it holds -- adds the splits in
// split order (its own from TMEM; with two splits it reads the other's slot straight
// from L2, with more it copies the other slots into the (now idle) operand ring with
// bulk copies), writes C and zeroes the counter.  No warp waits
// for another one, and the sum does not depend on the order of arrival.
// Returns false when the bulk copies did not complete in time (or could not fit).
// ahead / peeked: with S == 2, a warp that saw the other split's count while its own
// accumulator was still being computed has the first kTailAhead chunks of the other
// partial in `ahead` already and is the last (peeked).
template <int BN>
__device__ __forceinline__ bool pair_tail_epilogue(const GemmArgs &p, const CUtensorMap *tmC, uint32_t taddr,
                                                   uint32_t stage_smem, uint32_t stage_bytes, uint32_t red_bar,
                                                   int h, int split, uint32_t rank, int q, int lane, int x0,
                                                   int row0, bool bf16, uint32_t cbuf, int &nst,
                                                   uint32_t &red_phase, uint64_t lim, bool peeked,
                                                   float4 (&ahead)[kTailAhead][8]) {
    const int S = p.tail_splits;
    const int tt = h / S;  // leftover tile
    unsigned *ctr = pair_tail_counter(p, h, rank, q);
    unsigned last = peeked ? 1u : 0u;
    if (!peeked) {
        if (lane == 0) {
            unsigned seen;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(ctr) : "memory");
            last = seen + 1u == static_cast<unsigned>(S) ? 1u : 0u;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
    }
    if (!last) {
        float *mine = pair_tail_slot<BN>(p, h, rank, q);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c, r);
            tmem_ld_wait();
            float4 *dst = reinterpret_cast<float4 *>(mine + c * 32) + lane;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                __stcg(dst + 32 * j, make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) last = atomicAdd(ctr, 1u) + 1u == static_cast<unsigned>(S) ? 1u : 0u;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) return true;
    }
    __threadfence();
    if (lane == 0) *ctr = 0u;  // every split has arrived: ready for the next launch
    if (S == 2) {
        // One other partial: read it straight from L2, kTailAhead chunks ahead of the
        // sums (the loop is unrolled, so the in-flight chunks stay in registers), and add
        // it to this warp's own accumulator; own + other is the same sum whichever split
        // this warp holds.
        constexpr int kChunks = BN / 32;
        const float4 *oth = reinterpret_cast<const float4 *>(pair_tail_slot<BN>(p, tt * 2 + (split ^ 1), rank, q)) + lane;
        if (!peeked) pair_tail_load_ahead(oth, kChunks, ahead);
#pragma unroll
        for (int ci = 0; ci < kChunks; ++ci) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + 32 * ci, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 o = ahead[ci % kTailAhead][j];
                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + o.x);
                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + o.y);
                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + o.z);
                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + o.w);
            }
            if (ci + kTailAhead < kChunks) {
#pragma unroll
                for (int j = 0; j < 8; ++j) ahead[ci % kTailAhead][j] = __ldcg(oth + (ci + kTailAhead) * 256 + 32 * j);
            }
            store_chunk_tma(tmC, cbuf, nst++, r, bf16, x0 + 32 * ci, row0, lane);
        }
        return true;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");  // the other splits' stores, for the bulk copies
    // The other splits' slots come in through a ring of buffers in this warp's quarter of
    // the operand ring, 64 columns (32 KB / 4 of a 256-wide slot) at a time, one mbarrier
    // per buffer: the sums of one group overlap the copies of the next ones.
    const int others = S - 1;
    constexpr uint32_t kGroupBytes = 64u * 128u;  // 64 columns x 32 rows of fp32
    const uint32_t buf_bytes = static_cast<uint32_t>(others) * kGroupBytes;
    int nbuf = static_cast<int>(stage_bytes / buf_bytes);
    nbuf = nbuf > kTailBufs ? kTailBufs : nbuf;
    if (nbuf < 1) return false;  // the host plans no split count whose copies do not fit
    constexpr int kGroups = (BN + 63) / 64;
    auto issue = [&](int g) {  // lane 0: the copies of group g into buffer g % nbuf
        const int b = g % nbuf;
        const int cols = BN - 64 * g < 64 ? BN - 64 * g : 64;
        const uint32_t bytes = static_cast<uint32_t>(cols) * 128u;
        mbar_arrive_expect_tx(red_bar + 8u * b, bytes * static_cast<uint32_t>(others));
        int o = 0;
        for (int s2 = 0; s2 < S; ++s2) {
            if (s2 == split) continue;
            const float *src = pair_tail_slot<BN>(p, tt * S + s2, rank, q) + 64 * 32 * g;
            bulk_load(stage_smem + static_cast<uint32_t>(b) * buf_bytes + static_cast<uint32_t>(o++) * kGroupBytes,
                      src, bytes, red_bar + 8u * b);
        }
    };
    if (lane == 0)
        for (int g = 0; g < nbuf && g < kGroups; ++g) issue(g);
#pragma unroll 1
    for (int g = 0; g < kGroups; ++g) {
        const int b = g % nbuf;
        if (!warp_wait(red_bar + 8u * b, (red_phase >> b) & 1u, lim, lane)) return false;
        red_phase ^= 1u << b;
        const uint32_t buf = stage_smem + static_cast<uint32_t>(b) * buf_bytes + static_cast<uint32_t>(lane) * 16u;
        const int cols = BN - 64 * g < 64 ? BN - 64 * g : 64;
#pragma unroll 1
        for (int cc = 0; cc < cols; cc += 32) {
            const int c = 64 * g + cc;
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c, r);
            tmem_ld_wait();
            // the S terms in split order: this warp's own (r) at position `split`
            float acc[32];
            int o = 0;
            auto add_other = [&](bool first) {
                const uint32_t src = buf + static_cast<uint32_t>(o++) * kGroupBytes + static_cast<uint32_t>(cc) * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4 v;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                 : "r"(src + static_cast<uint32_t>(j) * 512u));
                    if (first) {
                        acc[4 * j] = v.x; acc[4 * j + 1] = v.y; acc[4 * j + 2] = v.z; acc[4 * j + 3] = v.w;
                    } else {
                        acc[4 * j] += v.x; acc[4 * j + 1] += v.y; acc[4 * j + 2] += v.z; acc[4 * j + 3] += v.w;
                    }
                }
            };
            if (split == 0) {
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(r[e]);
            } else {
                add_other(true);
                for (int s2 = 1; s2 < split; ++s2) add_other(false);
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] += __uint_as_float(r[e]);
            }
            for (int s2 = split + 1; s2 < S; ++s2) add_other(false);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(acc[e]);
            store_chunk_tma(tmC, cbuf, nst++, r, bf16, x0 + c, row0, lane);
        }
        __syncwarp();  // every lane has read buffer b
        if (lane == 0 && g + nbuf < kGroups) {
            fence_proxy_async_smem();  // those shared-memory reads, before the copies overwrite them
            issue(g + nbuf);
        }
    }
    return true;
}

// KSPLIT: the launch's last round is split in K (p.tail_splits >= 2); the other form
// of the kernel has none of that code.
template <int BN, int LAYOUT, bool KSPLIT>
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
    // kTailBufs per epilogue warp: bulk copies of a k-split tail's partials
    constexpr int kRedBars = KSPLIT ? Cfg::EPI_WARPS * kTailBufs : 0;
    uint64_t *red_bar = bars + 2 * S + 5;
    volatile uint32_t *ctrl = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 5 + kRedBars);

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
        for (int w = 0; w < kRedBars; ++w) mbar_init(smem_u32(&red_bar[w]), 1);
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
                int tile, m_tile, n_tile, n_off, width, k0, kn, split;
                pair_item<BN, KSPLIT>(item, p, tile, m_tile, n_tile, n_off, width, k0, kn, split);
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
                for (int i = 0; i < kn; ++i) {
                    if (!mbar_wait_for(empty0 + 8u * s, phase ^ 1u, lim)) {
                        record_status(p.status, kSiteProducer | static_cast<int>(rank << 4) | (issued << 8));
                        ctrl[1] = 1;
                        stop = true;
                        break;
                    }
                    if ((i & 7) == 0 && ctrl[1]) { stop = true; break; }  // another role gave up
                    const int kt = (p.stagger && split < 0) ? ((start + i) & (nK - 1)) : k0 + i;
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
                const uint32_t idesc = (item < p.tail_start || KSPLIT) ? idesc_full : idesc_half;
                int tile, m_tile, n_tile, n_off, width, k0, kn, split;
                pair_item<BN, KSPLIT>(item, p, tile, m_tile, n_tile, n_off, width, k0, kn, split);
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
                for (int i = 0; i < kn; ++i) {
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
        uint32_t red_phase = 0;
        // this warp's quarter of the operand ring, which a k-split tail item (always its
        // pair's last item) reuses once its own MMAs have completed
        const uint32_t ring_quarter = (static_cast<uint32_t>(S) * Cfg::STAGE_BYTES / Cfg::EPI_WARPS) & ~1023u;
        const uint32_t stage_smem = smem_u32(smA) + static_cast<uint32_t>(q) * ring_quarter;
        int j = 0;
        for (int item = pair; item < num_items; item += num_pairs, ++j) {
            const int b = j & 1;
            const uint32_t acc_phase = static_cast<uint32_t>((j >> 1) & 1);
            bool peeked = false;
            float4 ahead[kTailAhead][8];
            if constexpr (KSPLIT) {
                // a two-way split item: while its accumulator is being computed, watch the
                // other split's count, and once that split has published its partial, start
                // loading the partial's first chunks
                if (p.tail_splits == 2 && item >= p.tail_start) {
                    const int h = item - p.tail_start;
                    const int st = warp_wait_or_count(smem_u32(&acc_full[b]), acc_phase,
                                                      pair_tail_counter(p, h, rank, q), 1u, 4 * lim, lane);
                    if (st == 2) {
                        peeked = true;
                        __threadfence();
                        const float4 *oth = reinterpret_cast<const float4 *>(
                                                pair_tail_slot<BN>(p, h ^ 1, rank, q)) + lane;
                        pair_tail_load_ahead(oth, BN / 32, ahead);
                    }
                }
            }
            if (!warp_wait(smem_u32(&acc_full[b]), acc_phase, 4 * lim, lane)) {
                if (lane == 0) {
                    record_status(p.status, kSiteEpilogue | static_cast<int>(rank << 4) | (j << 8));
                    ctrl[1] = 1;
                }
                break;
            }
            tc_fence_after();
            int tile, m_tile, n_tile, n_off, width, k0, kn, split;
            pair_item<BN, KSPLIT>(item, p, tile, m_tile, n_tile, n_off, width, k0, kn, split);
            const int row0 = m_tile * Cfg::BM + static_cast<int>(rank) * Cfg::CTA_M + q * 32;  // this warp's rows
            const int n0 = n_tile * BN + n_off;
            const bool bf16 = ((p.idesc_flags >> 7) & 7u) == 1u;
            const uint32_t taddr =
                tmem_base + static_cast<uint32_t>(b * BN) + (static_cast<uint32_t>(q * 32) << 16);
            if constexpr (KSPLIT) {
                if (split >= 0) {
                    const bool ok = pair_tail_epilogue<BN>(p, &tmC, taddr, stage_smem, ring_quarter,
                                                           smem_u32(&red_bar[q * kTailBufs]), item - p.tail_start,
                                                           split, rank, q, lane, n0, row0, bf16, cbuf, nst,
                                                           red_phase, lim, peeked, ahead);
                    // the accumulator was read for the last time: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[b]), 0));
                        if (!ok) {
                            record_status(p.status, kSiteEpilogue | 0x40 | static_cast<int>(rank << 4) | (j << 8));
                            ctrl[1] = 1;
                        }
                    }
                    if (!ok) break;
                    continue;
                }
            }
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
