// gemm_kernel.cuh -- tcgen05 fp16 GEMM kernel template, one CTA per output tile.
//
// C[M][N] = A[M][K] . B[K][N]; fp16 operands, fp32 accumulation in tensor memory,
// fp16 output.  The CTA tile BM x BN is a template parameter so that the host can
// pick it from the problem shape ("Beating hipBLASLt on a Gaming GPU", section
// "The part that actually mattered": tile shape as a compile-time kernel
// parameter, one of several, chosen per launch).
//
// Roles inside a 128-thread CTA:
//   warp 0, lane 0 : TMA producer.  Per k-tile: wait for the ring slot to be free,
//                    arm its "full" barrier with the byte count, issue TMA loads of
//                    A[BM x 64] (K-major, 128-byte swizzle) and B[64 x BN] (N
//                    contiguous, 128-byte swizzle, one 64-column box at a time).
//   warp 1, lane 0 : MMA issuer.  Per k-tile: wait "full", issue 4 x
//                    tcgen05.mma (K = 16 each) into the TMEM accumulator, then
//                    tcgen05.commit to the slot's "empty" barrier.  After the last
//                    k-tile, commit to "acc_full".
//   all 4 warps    : epilogue.  Wait "acc_full", tcgen05.ld 32 columns at a time
//                    from the warp's TMEM lane quarter, round to fp16, store C.
//
// The k-loop start stagger (FlyDSL pull request "Speed up the RDNA3 GEMM up to
// 1.85x by choosing the tile from the shape", "Changes" and third commit message)
// starts CTA b at k-tile (b * stride) & (nK - 1) and wraps with the same mask; the
// host enables it only when nK is a power of two.
//
// CTAs are rasterised in bands of `raster_group` m-tiles so that the A and B
// panels in flight at any moment stay resident in L2.
//
// Every wait is bounded by a deadline; on expiry the kernel records a code in
// the device status word, drains its own TMA copies (bounded again), frees its
// TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace sdt {

constexpr int kBK = 64;  // k-depth per ring slot: one 128-byte swizzle row of fp16

struct GemmArgs {
    __half *C;
    int M, N, K;
    int num_m_tiles, num_n_tiles, num_k_tiles;
    int stages;           // ring depth used by this launch (<= the tile's maximum)
    int stagger;          // 1: per-CTA k-loop start stagger (num_k_tiles is a power of two)
    int stagger_stride;   // k-tiles between the start points of consecutive CTAs
    int raster_group;     // m-tiles per raster band
    unsigned long long timeout_ns;
    int *status;          // device status word (first error code wins)
    int max_ctas;         // persistent kernels: grid size cap (one CTA per SM); host-side only
    // split-K (blockIdx.y = split): k-tiles [split*k_per_split, ...) of each output tile
    int splits;
    int k_per_split;
    int splitk_reduce_in_kernel;  // 1: the last CTA of a tile sums the partials and writes C
    float *partials;      // [splits][num_m_tiles*BM][num_n_tiles*BN] fp32 (two-CTA tail: one slot per item)
    unsigned *counters;   // [num_m_tiles * num_n_tiles], zero between calls (two-CTA tail: 8 per tile)
    // two-CTA tiles: work items [0, tail_start) are whole tiles; items
    // [tail_start, num_items) cover tiles tail_start ...: two column halves per tile
    // (tail_splits == 0), or tail_splits k-ranges per tile whose fp32 partials go to
    // `partials` and are counted on `counters` (tail_splits >= 2)
    int tail_start;
    int num_items;
    int tail_splits;
    int tail_long;          // k-split tail: k-tiles of split 0 (the others share the rest evenly); 0: all even
    int ldc;                // row stride of C in elements
    uint32_t idesc_flags;   // instruction-descriptor bits: accumulator, operand types, operand majors
    int c_trans;            // 1: element (r, c) of this problem is C[c * ldc + r] (operands swapped)
};

// Operand layouts, a template parameter of every GEMM kernel: bit 0 set means A is
// stored K x M (M contiguous, "transposed A"); bit 1 set means B is stored N x K
// (K contiguous, "transposed B").  LAYOUT 0 is row-major A (M x K) and B (K x N).
template <int LAYOUT>
struct OperandLayout {
    static constexpr bool A_MN = (LAYOUT & 1) != 0;  // A tile is MN-major in shared memory
    static constexpr bool B_MN = (LAYOUT & 2) == 0;  // B tile is MN-major in shared memory
};

// One operand tile of ROWS rows (M or N) x 64 K-elements for k-tile kt.
// MN-major operand (rows contiguous in memory): ceil(ROWS/64) TMA boxes of 64 x 64, box c
// covering rows r0+64c .. +63 and landing at dst + 8 KB * c as 64 k-rows of 128 B
// (canonical MN-major 128 B swizzle: 64-element chunks 8 KB apart).  K-major operand
// (K contiguous): ROWS/KBOX boxes of 64 x KBOX (KBOX = ROWS when the whole tile is one
// box), landing as consecutive 128-byte rows (canonical K-major 128 B swizzle: 8-row
// groups 1024 B apart).
template <bool PAIR, bool MN, int ROWS, int KBOX>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap *map, uint32_t bar, int kt, int r0) {
    if constexpr (MN) {
        // (a width that is not a multiple of 64 takes a last whole box; its extra
        // columns land in the unused part of the last 64-column block)
#pragma unroll
        for (int c = 0; c < (ROWS + 63) / 64; ++c) {
            if (PAIR) tma_load_2d_pair(dst + c * 8192, map, bar, r0 + 64 * c, kt * kBK);
            else tma_load_2d(dst + c * 8192, map, bar, r0 + 64 * c, kt * kBK);
        }
    } else {
        static_assert(ROWS % KBOX == 0, "K-major tile must be whole boxes");
#pragma unroll
        for (int c = 0; c < ROWS / KBOX; ++c) {
            if (PAIR) tma_load_2d_pair(dst + c * KBOX * 128, map, bar, kt * kBK, r0 + KBOX * c);
            else tma_load_2d(dst + c * KBOX * 128, map, bar, kt * kBK, r0 + KBOX * c);
        }
    }
}

// Shared-memory matrix descriptor of a staged operand tile and its advance (in
// 16-byte units) per K = 16 MMA step: +32 B along a K-major row, +2 KB (16 k-rows)
// for an MN-major tile.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base) {
    return MN ? smem_desc_sw128(base, 8192, 1024) : smem_desc_sw128(base, 16, 1024);
}
template <bool MN>
__host__ __device__ constexpr uint64_t operand_k_step() {
    return MN ? 128ull : 2ull;
}

// Instruction descriptor for an M x N MMA with the runtime type/major bits.
__device__ __forceinline__ uint32_t idesc_for(uint32_t flags, int M, int N) {
    return flags | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Stores 32 fp32 accumulator columns of one C row as fp16/bf16, 16 bytes at a time,
// skipping vectors at or beyond column limit `ncols` (a multiple of 8).
__device__ __forceinline__ void store_row32(void *crow, const uint32_t (&r)[32], int ncols, bool bf16) {
    uint32_t h[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        const float lo = __uint_as_float(r[2 * t]), hi = __uint_as_float(r[2 * t + 1]);
        if (bf16) {
            __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
            h[t] = *reinterpret_cast<uint32_t *>(&v);
        } else {
            __half2 v = __floats2half2_rn(lo, hi);
            h[t] = *reinterpret_cast<uint32_t *>(&v);
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(crow);
#pragma unroll
    for (int v = 0; v < 4; ++v)
        if (8 * v + 8 <= ncols) dst[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
}

// C through shared memory and TMA stores (persistent and two-CTA kernels).  Each
// epilogue warp owns two staging buffers of 32 rows x 32 columns of 16-bit C (2 KB),
// used alternately; a buffer holds the box of a C tensor map with a 32 x 32 box and
// the 64-byte swizzle: row r's 16-byte chunk c sits at chunk c ^ ((r >> 1) & 3) of
// its 64-byte row, so the warp's 16-byte writes of one chunk index reach 32 distinct
// banks in every 8-lane phase.  The TMA writes whole 64-byte row pieces of C and
// drops rows and columns outside C, so ragged edges need no masks.
constexpr int kCStageBytes = 32 * 32 * 2;

// Lane = row: its 32 fp32 accumulator columns -> fp16/bf16 -> staging buffer (nst & 1)
// -> one TMA store of the warp's 32 x 32 box at (x, y).  Lane 0 issues the store and
// first waits until the store that last used the buffer has read it.
__device__ __forceinline__ void store_chunk_tma(const CUtensorMap *tmC, uint32_t buf0, int nst,
                                                const uint32_t (&r)[32], bool bf16, int x, int y, int lane) {
    uint32_t h[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        const float lo = __uint_as_float(r[2 * t]), hi = __uint_as_float(r[2 * t + 1]);
        if (bf16) {
            __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
            h[t] = *reinterpret_cast<uint32_t *>(&v);
        } else {
            __half2 v = __floats2half2_rn(lo, hi);
            h[t] = *reinterpret_cast<uint32_t *>(&v);
        }
    }
    const uint32_t buf = buf0 + static_cast<uint32_t>(nst & 1) * kCStageBytes;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    const uint32_t row = buf + static_cast<uint32_t>(lane) * 64u;
    const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((static_cast<uint32_t>(c) ^ sw) << 4)),
                     "r"(h[4 * c]), "r"(h[4 * c + 1]), "r"(h[4 * c + 2]), "r"(h[4 * c + 3])
                     : "memory");
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmC, buf, x, y);
        bulk_commit_group();
    }
}

// One fp32 value -> fp16 or bf16 bits (round to nearest even).
__device__ __forceinline__ uint16_t f32_to_16(float v, bool bf16) {
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

// Eight fp32 values -> eight fp16 or bf16 (round to nearest even), packed for one 16-byte store.
__device__ __forceinline__ uint4 pack8_f32(const float4 &a, const float4 &b, bool bf16) {
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t h[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if (bf16) {
            __nv_bfloat162 x = __floats2bfloat162_rn(v[2 * t], v[2 * t + 1]);
            h[t] = *reinterpret_cast<uint32_t *>(&x);
        } else {
            __half2 x = __floats2half2_rn(v[2 * t], v[2 * t + 1]);
            h[t] = *reinterpret_cast<uint32_t *>(&x);
        }
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

template <int BM, int BN>
struct TileCfg {
    static constexpr int A_BYTES = BM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int B_BOX_BYTES = 64 * kBK * 2;  // one 64-column box of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;  // fp32 accumulator columns (power of two, >= 32)
    static constexpr int THREADS = 128;
    static constexpr int ALIGN_SLACK = 1024;           // dynamic smem base rounded up to 1024 B
    static constexpr int CTRL_BYTES = 512;             // barriers + TMEM address + flags
    __host__ __device__ static constexpr int smem_bytes(int stages) {
        return ALIGN_SLACK + stages * STAGE_BYTES + CTRL_BYTES;
    }
    static_assert(BM == 64 || BM == 128, "BM must be 64 or 128");
    static_assert(BN == 16 || BN == 32 || BN == 64 || BN == 128 || BN == 256, "BN must be 16 .. 256");
};

__device__ __forceinline__ void record_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// SPLIT: the CTA accumulates only its split's k-tiles and writes an fp32 partial
// tile to p.partials[split]; with p.splitk_reduce_in_kernel the last CTA of the
// output tile to finish (per-tile arrival counter) sums all partials in split
// order and writes the fp16 tile, then resets the counter to zero.
template <int BM, int BN, bool SPLIT, int LAYOUT>
__global__ void __launch_bounds__(128, 1)
    gemm_f16_tile_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const GemmArgs p) {
    using Cfg = TileCfg<BM, BN>;
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
    uint64_t *acc_full = bars + 2 * S;
    volatile uint32_t *ctrl = reinterpret_cast<volatile uint32_t *>(bars + 2 * S + 1);
    // ctrl[0]: TMEM base address   ctrl[1]: error flag   ctrl[2]: k-tiles issued by TMA
    // ctrl[3]: split-K, this CTA is the last of its tile

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Output tile of this CTA (banded raster order).
    const int lin = blockIdx.x;
    const int per_band = p.raster_group * p.num_n_tiles;
    const int band = lin / per_band;
    const int first_m = band * p.raster_group;
    const int band_m = min(p.num_m_tiles - first_m, p.raster_group);
    const int in_band = lin - band * per_band;
    const int m_tile = first_m + in_band % band_m;
    const int n_tile = in_band / band_m;
    const int m0 = m_tile * BM;
    const int n0 = n_tile * BN;
    const int split = SPLIT ? static_cast<int>(blockIdx.y) : 0;
    const int k_first = SPLIT ? split * p.k_per_split : 0;
    const int nK = SPLIT ? min(p.k_per_split, p.num_k_tiles - k_first) : p.num_k_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(acc_full), 1);
        ctrl[1] = 0;
        ctrl[2] = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(&ctrl[0])), Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = ctrl[0];
    griddep_launch_dependents();
    griddep_wait();  // the previous kernel's writes (A, B, C) are visible from here on

    const uint64_t t_start = global_timer_ns();
    const uint64_t deadline = t_start + p.timeout_ns;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        const bool stagger = !SPLIT && p.stagger;
        const int start = stagger
            ? static_cast<int>((static_cast<uint32_t>(lin) * static_cast<uint32_t>(p.stagger_stride)) &
                               static_cast<uint32_t>(nK - 1))
            : 0;
        int s = 0;
        uint32_t phase = 0;
        // per-slot addresses are fixed offsets from slot 0: the loop adds instead of
        // recomputing them, and reads the error flag only every eighth k-tile (this
        // single thread's instruction count per k-tile sets the pace of small tiles)
        const uint32_t empty0 = smem_u32(&empty[0]), full0 = smem_u32(&full[0]);
        const uint32_t smA0 = smem_u32(smA), smB0 = smem_u32(smB);
        int i = 0;
// (the k-loops of the producer and MMA threads are unrolled by four: these single
// threads set the pace of a k-tile, and the unrolled loop issues fewer instructions)
#pragma unroll 4
        for (; i < nK; ++i) {
            if (!mbar_wait(empty0 + 8u * s, phase ^ 1u, deadline)) {
                record_status(p.status, kSiteProducer);
                ctrl[1] = 1;
                break;
            }
            if ((i & 7) == 0 && ctrl[1]) break;
            const int kt = k_first + (stagger ? ((start + i) & (nK - 1)) : i);
            const uint32_t fb = full0 + 8u * s;
            mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
            load_operand<false, L::A_MN, BM, BM>(smA0 + static_cast<uint32_t>(s) * Cfg::A_BYTES, &tmA, fb, kt, m0);
            // (tiles narrower than 64 columns take K-major B only: boxes of BN rows)
            load_operand<false, L::B_MN, BN, (BN < 64 ? BN : 64)>(smB0 + static_cast<uint32_t>(s) * Cfg::B_BYTES,
                                                                 &tmB, fb, kt, n0);
            if (++s == S) { s = 0; phase ^= 1u; }
        }
        ctrl[2] = i;  // k-tiles issued: read by the drain after an error
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = idesc_for(p.idesc_flags, BM, BN);
        constexpr uint64_t a_step = operand_k_step<L::A_MN>(), b_step = operand_k_step<L::B_MN>();
        int s = 0;
        uint32_t phase = 0;
        // slot s's descriptors are slot 0's plus s stages (the start address field counts
        // 16-byte units and shared memory stays below 2^18 bytes)
        const uint64_t a_desc0 = operand_desc<L::A_MN>(smem_u32(smA));
        const uint64_t b_desc0 = operand_desc<L::B_MN>(smem_u32(smB));
        const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
#pragma unroll 4
        for (int i = 0; i < nK; ++i) {
            if (!mbar_wait(full0 + 8u * s, phase, deadline)) {
                record_status(p.status, kSiteMma);
                ctrl[1] = 1;
                break;
            }
            tc_fence_after();
            const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(s) * (Cfg::A_BYTES >> 4);
            const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(s) * (Cfg::B_BYTES >> 4);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                umma_f16(tmem_d, a_desc + a_step * kk, b_desc + b_step * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
            umma_commit(empty0 + 8u * s);
            if (++s == S) { s = 0; phase ^= 1u; }
        }
        umma_commit(smem_u32(acc_full));
    }
    __syncwarp();

    // ---------------- epilogue: TMEM -> registers -> fp16 -> global ----------------
    const bool acc_ok = mbar_wait_sleepy(smem_u32(acc_full), 0, t_start + 3ull * p.timeout_ns);
    if (!acc_ok) {
        record_status(p.status, kSiteEpilogue);
        ctrl[1] = 1;
    }
    tc_fence_after();
    {
        // Accumulator row r sits in TMEM lane r for M = 128; for M = 64 rows
        // 16q .. 16q+15 sit in lanes 32q .. 32q+15 of lane quarter q.
        const int row = (BM == 128) ? (warp * 32 + lane) : (warp * 16 + lane);
        const bool row_valid = ((BM == 128) || (lane < 16)) && (m0 + row < p.M);
        const uint32_t taddr_row = tmem_d + (static_cast<uint32_t>(warp * 32) << 16);
        const bool bf16 = ((p.idesc_flags >> 7) & 7u) == 1u;
        uint16_t *crow = reinterpret_cast<uint16_t *>(p.C) + static_cast<size_t>(m0 + row) * p.ldc + n0;
        // partial planes are [splits][num_m_tiles*BM][num_n_tiles*BN]: whole tiles, so the
        // 32-column stores below need no column mask on ragged shapes
        const size_t Mp = static_cast<size_t>(p.num_m_tiles) * BM, Np = static_cast<size_t>(p.num_n_tiles) * BN;
        float *prow = SPLIT ? p.partials + (static_cast<size_t>(split) * Mp + m0 + row) * Np + n0 : nullptr;
        constexpr int CH = BN < 32 ? BN : 32;  // accumulator columns per TMEM load
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
            uint32_t r[32];
            if (CH == 32) tmem_ld_32x32b_x32(taddr_row + c, r);
            else tmem_ld_32x32b_x16(taddr_row + c, r);
            tmem_ld_wait();
            if (SPLIT) {
                if (row_valid && acc_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(prow + c);
#pragma unroll
                    for (int t = 0; t < CH / 4; ++t) dst[t] = make_uint4(r[4 * t], r[4 * t + 1], r[4 * t + 2], r[4 * t + 3]);
                }
                continue;
            }
            if (!(row_valid && acc_ok)) continue;
            if (p.c_trans) {
                // swapped operands: this accumulator row is column m0 + row of C; lanes hold
                // consecutive rows, so each store instruction writes 32 neighbouring elements
                uint16_t *ccol = reinterpret_cast<uint16_t *>(p.C) + m0 + row;
#pragma unroll
                for (int t = 0; t < CH; ++t)
                    if (n0 + c + t < p.N)
                        ccol[static_cast<size_t>(n0 + c + t) * p.ldc] = f32_to_16(__uint_as_float(r[t]), bf16);
            } else {
                store_row32(crow + c, r, p.N - (n0 + c), bf16);
            }
        }
    }
    tc_fence_before();
    if (SPLIT && p.splitk_reduce_in_kernel) {
        // Publish this split's partial, then count arrivals on the tile; the last CTA
        // to arrive sums every split's partial in split order (so the result does not
        // depend on arrival order), writes C, and resets the counter for the next call.
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned prev = atomicAdd(&p.counters[lin], 1u);
            ctrl[3] = (prev == static_cast<unsigned>(p.splits - 1)) ? 1u : 0u;
        }
        __syncthreads();
        if (ctrl[3]) {
            __threadfence();
            const int vrows = min(BM, p.M - m0);  // rows of the tile inside C
            if (vrows > 0 && !ctrl[1]) {
                // The tile's rows inside C, 8 consecutive columns per thread and step (a
                // warp reads whole sectors of a partial row), up to four steps per pass:
                // every load of a split in a pass is issued before any of it is used.
                const size_t Np = static_cast<size_t>(p.num_n_tiles) * BN;
                const size_t plane = static_cast<size_t>(p.num_m_tiles) * BM * Np;
                const float *src0 = p.partials + static_cast<size_t>(m0) * Np + n0;
                const bool bf16 = ((p.idesc_flags >> 7) & 7u) == 1u;
                const int total = vrows * BN;
                constexpr int STEP = Cfg::THREADS * 8;
#pragma unroll 1
                for (int e0 = static_cast<int>(threadIdx.x) * 8; e0 < total; e0 += 4 * STEP) {
                    float4 acc[8];
#pragma unroll 2
                    for (int sp = 0; sp < p.splits; ++sp) {
                        float4 x[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int e = e0 + i * STEP;
                            const float *src = src0 + sp * plane + static_cast<size_t>(e / BN) * Np + (e % BN);
                            if (e < total) {
                                x[2 * i] = __ldcg(reinterpret_cast<const float4 *>(src));
                                x[2 * i + 1] = __ldcg(reinterpret_cast<const float4 *>(src + 4));
                            } else {
                                x[2 * i] = x[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (sp == 0) {
                                acc[i] = x[i];
                            } else {
                                acc[i].x += x[i].x; acc[i].y += x[i].y; acc[i].z += x[i].z; acc[i].w += x[i].w;
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int e = e0 + i * STEP;
                        if (e >= total) continue;
                        const int r = e / BN, c = e % BN;
                        if (n0 + c >= p.N) continue;
                        if (p.c_trans) {
                            const float v[8] = {acc[2 * i].x, acc[2 * i].y, acc[2 * i].z, acc[2 * i].w,
                                                acc[2 * i + 1].x, acc[2 * i + 1].y, acc[2 * i + 1].z, acc[2 * i + 1].w};
                            uint16_t *ccol = reinterpret_cast<uint16_t *>(p.C) + m0 + r;
#pragma unroll
                            for (int t = 0; t < 8; ++t)
                                if (n0 + c + t < p.N) ccol[static_cast<size_t>(n0 + c + t) * p.ldc] = f32_to_16(v[t], bf16);
                        } else {  // N % 8 == 0 unless transposed
                            uint16_t *crow = reinterpret_cast<uint16_t *>(p.C) + static_cast<size_t>(m0 + r) * p.ldc + n0;
                            *reinterpret_cast<uint4 *>(crow + c) = pack8_f32(acc[2 * i], acc[2 * i + 1], bf16);
                        }
                    }
                }
            }
            if (threadIdx.x == 0) atomicExch(&p.counters[lin], 0u);
        }
    }
    __syncthreads();

    if (threadIdx.x == 0 && ctrl[1]) {
        // Drain: wait (bounded) for every TMA copy this CTA issued and may not have seen land.
        const int issued = static_cast<int>(ctrl[2]);
        const uint64_t drain_deadline = global_timer_ns() + p.timeout_ns;
        for (int i = max(0, issued - S); i < issued; ++i) {
            if (!mbar_wait(smem_u32(&full[i % S]), static_cast<uint32_t>((i / S) & 1), drain_deadline)) {
                record_status(p.status, kSiteDrain);
                break;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_d, Cfg::TMEM_COLS);
    }
}

// Sums the fp32 partials [splits][Mp][Np] in split order and writes C [M][N] (row
// stride ldc, fp16 or bf16): the separate-kernel reduction of split-K; each thread
// handles 8 consecutive columns of one row.
__global__ void splitk_reduce_kernel(const float *__restrict__ partials, uint16_t *__restrict__ C, int64_t M,
                                     int64_t N, int64_t Mp, int64_t Np, int64_t ldc, int splits, int bf16);
// The same for swapped operands: element (r, c) of the problem goes to C[c * ldc + r];
// one element per thread, consecutive threads on consecutive r (coalesced stores).
__global__ void splitk_reduce_trans_kernel(const float *__restrict__ partials, uint16_t *__restrict__ C,
                                           int64_t M, int64_t N, int64_t Mp, int64_t Np, int64_t ldc, int splits,
                                           int bf16);

// Host-side launchers, instantiated per ladder tile and layout (gemm_t*.cu).  The
// ladder's launchers take the C map of the persistent and two-CTA kernels' TMA
// stores; the one-CTA kernel stores C directly and ignores it.
template <int BM, int BN, int LAYOUT>
int launch_gemm_tile(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &args,
                     cudaStream_t stream);
template <int BM, int BN, int LAYOUT>
int launch_gemm_tile_split(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &args,
                           cudaStream_t stream);

}  // namespace sdt
