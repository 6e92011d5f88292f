// gemm_host.cu -- host side of gemm_f16: the tile ladder, feasible_tiles,
// pick_tile, the frozen tune table, the opt-in measured sweep, TMA tensor maps
// and the C-ABI entry points.
//
// Tile selection follows the FlyDSL pull request "Speed up the RDNA3 GEMM up to
// 1.85x by choosing the tile from the shape", section "Changes": a heuristic
// (pick_tile) that needs no GPU and measures nothing chooses among the tiles that
// feasible_tiles admits; an opt-in measured sweep (SDT_AUTOTUNE=1) times every
// feasible tile, and a sweep's result can be frozen into a table
// (SDT_TUNE_TABLE) that overrides the heuristic.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cerrno>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "gemm_kernel.cuh"
#include "gemm_persistent.cuh"
#include "gemm_pair.cuh"
#include "gemm_streamk.cuh"
#include "host_common.cuh"

namespace sdt {

using LaunchFn = int (*)(const CUtensorMap &, const CUtensorMap &, const GemmArgs &, cudaStream_t);
// The ladder's launchers also take the C map (TMA stores of the persistent and two-CTA kernels).
using TileLaunchFn = int (*)(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const GemmArgs &,
                             cudaStream_t);

// Split-K launchers of the one-CTA-per-tile ladder rungs, in ladder order, per operand
// layout (null: no split-K form).
#define SDT_SPLIT4_(BM, BN)                                                                        \
    {&launch_gemm_tile_split<BM, BN, 0>, &launch_gemm_tile_split<BM, BN, 1>,                       \
     &launch_gemm_tile_split<BM, BN, 2>, &launch_gemm_tile_split<BM, BN, 3>}
static const LaunchFn kSplitLaunch[][4] = {
    SDT_SPLIT4_(64, 64),   SDT_SPLIT4_(64, 128),  SDT_SPLIT4_(128, 64),  SDT_SPLIT4_(128, 128),
    SDT_SPLIT4_(128, 256), {nullptr, nullptr, nullptr, nullptr},     {nullptr, nullptr, nullptr, nullptr},
    {nullptr, nullptr, nullptr, nullptr},         {nullptr, nullptr, nullptr, nullptr},
    {nullptr, nullptr, nullptr, nullptr},         SDT_SPLIT4_(128, 16),  SDT_SPLIT4_(128, 32)};

// Stream-K launchers of the same rungs (null: no stream-K form).
#define SDT_STREAM4_(BM, BN)                                                                       \
    {&launch_gemm_streamk<BM, BN, 0>, &launch_gemm_streamk<BM, BN, 1>, &launch_gemm_streamk<BM, BN, 2>, \
     &launch_gemm_streamk<BM, BN, 3>}
static const LaunchFn kStreamLaunch[][4] = {
    SDT_STREAM4_(64, 64),   SDT_STREAM4_(64, 128),  SDT_STREAM4_(128, 64),  SDT_STREAM4_(128, 128),
    SDT_STREAM4_(128, 256), {nullptr, nullptr, nullptr, nullptr},       {nullptr, nullptr, nullptr, nullptr},
    {nullptr, nullptr, nullptr, nullptr},           {nullptr, nullptr, nullptr, nullptr},
    {nullptr, nullptr, nullptr, nullptr},           SDT_STREAM4_(128, 16),  SDT_STREAM4_(128, 32)};

// One rung of the tile ladder.  kt_cycles / fixed_cycles feed pick_tile's cost
// model: SM cycles one CTA of this tile spends per 64-deep k-tile when it has
// the SM to itself, and its per-CTA fixed cost (TMEM allocation, pipeline fill,
// epilogue).  They are fitted to the measured sweep of every feasible tile.
struct LadderTile {
    int BM, BN, cta_group, stages;
    const char *name;
    TileLaunchFn launch[4];  // per operand layout (bit 0: A transposed, bit 1: B transposed)
    int smem_per_stage;
    int smem_fixed;
    int tmem_cols;
    int threads;
    bool persistent;  // one CTA per SM walking tiles; accumulator double-buffered in TMEM
    // pick_tile cost model, fitted to the measured sweep of every feasible tile (us):
    //   fixed -- once per launch: the launch, the pipeline fill and the first
    //            `stages` k-tiles (issued as one burst)
    //   kt    -- per further k-tile on the busiest worker (CTA or CTA pair)
    //   round -- per round of tiles on one worker (a wave of co-resident CTAs, or
    //            a persistent worker's next tile): the exposed epilogue and refill
    //   bw    -- per k-tile of the whole grid's work divided by the workers the
    //            device holds: the share of the operand streaming that the L2
    //            does not overlap with the MMAs (large for the wide pair tile)
    //   share -- per CTA beyond the first on the busiest SM of a wave (tiles that
    //            fit two CTAs per SM)
    double fixed_us;
    double kt_us;
    double round_us;
    double bw_us;
    double share_us;
    bool candidate;   // considered by pick_tile (tiles dominated everywhere in the sweep are not)
    bool swap = false;  // skinny tile: runs C^T = op(B)^T . op(A)^T (gemm_ex forms only)
};

#define SDT_LAUNCH4_(FN, ...) {&FN<__VA_ARGS__, 0>, &FN<__VA_ARGS__, 1>, &FN<__VA_ARGS__, 2>, &FN<__VA_ARGS__, 3>}

#define SDT_TILE(BM_, BN_, STAGES_, NAME_, FIX_, KT_, RND_, BW_, SHR_, CAND_)                          \
    LadderTile {                                                                                   \
        BM_, BN_, 1, STAGES_, NAME_, SDT_LAUNCH4_(launch_gemm_tile, BM_, BN_),                     \
            TileCfg<BM_, BN_>::STAGE_BYTES, TileCfg<BM_, BN_>::ALIGN_SLACK + TileCfg<BM_, BN_>::CTRL_BYTES, \
            TileCfg<BM_, BN_>::TMEM_COLS, TileCfg<BM_, BN_>::THREADS, false, FIX_, KT_, RND_, BW_, SHR_, CAND_ \
    }

#define SDT_PTILE(BN_, STAGES_, NAME_, FIX_, KT_, RND_, BW_, CAND_)                                     \
    LadderTile {                                                                                   \
        128, BN_, 1, STAGES_, NAME_, SDT_LAUNCH4_(launch_gemm_persistent, BN_),                    \
            PersistentCfg<BN_>::STAGE_BYTES,                                                         \
            PersistentCfg<BN_>::ALIGN_SLACK + PersistentCfg<BN_>::C_STAGE_BYTES + PersistentCfg<BN_>::CTRL_BYTES, \
            PersistentCfg<BN_>::TMEM_COLS, PersistentCfg<BN_>::THREADS, true, FIX_, KT_, RND_, BW_, 0.0, CAND_ \
    }

#define SDT_STILE(BN_, STAGES_, NAME_, FIX_, KT_)                                                    \
    LadderTile {                                                                                   \
        128, BN_, 1, STAGES_, NAME_, SDT_LAUNCH4_(launch_gemm_tile, 128, BN_),                     \
            TileCfg<128, BN_>::STAGE_BYTES, TileCfg<128, BN_>::ALIGN_SLACK + TileCfg<128, BN_>::CTRL_BYTES, \
            TileCfg<128, BN_>::TMEM_COLS, TileCfg<128, BN_>::THREADS, false, FIX_, KT_, 0.0, 0.0, 0.0, false, true \
    }

#define SDT_PAIR(BN_, STAGES_, NAME_, FIX_, KT_, RND_, BW_, CAND_)                                      \
    LadderTile {                                                                                   \
        256, BN_, 2, STAGES_, NAME_, SDT_LAUNCH4_(launch_gemm_pair, BN_), PairCfg<BN_>::STAGE_BYTES, \
            PairCfg<BN_>::ALIGN_SLACK + PairCfg<BN_>::C_STAGE_BYTES + PairCfg<BN_>::CTRL_BYTES,    \
            PairCfg<BN_>::TMEM_COLS,                                                               \
            PairCfg<BN_>::THREADS, true, FIX_, KT_, RND_, BW_, 0.0, CAND_                                  \
    }

// Cost-model constants fitted on GB300 (152 SMs) by one non-negative least-squares
// fit, weighted by 1 / sqrt(time), over two cold-L2 sweeps of every feasible tile
// (bench.py --mode sweep) of the current kernels (persistent and two-CTA kernels with
// TMA stores of C): 43 shapes (the square sizes, the K-scan around 2048^2,
// rectangular, skinny and deep-K shapes) and a second measurement of the 15 square and
// K-scan ones.  The fitted model's pick is within 2.7 % of the best swept tile on
// every one of those shapes (0.14 % on average), and stays there with each shape
// left out of the fit in turn (python -m shape_driven_tile_gb300.costfit refits it).
static const LadderTile kLadder[] = {
    SDT_TILE(64, 64, 6, "64x64", 6.293, 0.22299, 2.473, 0.01095, 1.323, true),
    SDT_TILE(64, 128, 4, "64x128", 6.288, 0.24812, 2.152, 0.05457, 1.466, true),
    SDT_TILE(128, 64, 4, "128x64", 6.654, 0.24589, 1.764, 0.06153, 1.353, true),
    SDT_TILE(128, 128, 6, "128x128", 5.266, 0.21826, 4.685, 0.01681, 0.000, true),
    SDT_TILE(128, 256, 4, "128x256", 5.328, 0.30875, 5.201, 0.04317, 0.000, false),
    SDT_PTILE(128, 6, "p128x128", 9.292, 0.20648, 0.219, 0.01416, true),
    SDT_PTILE(256, 4, "p128x256", 9.295, 0.31192, 0.158, 0.03885, true),
    SDT_PAIR(128, 8, "2cta_256x128", 11.744, 0.23670, 0.275, 0.00779, false),
    SDT_PAIR(256, 6, "2cta_256x256", 11.060, 0.22789, 0.000, 0.10519, true),
    // 224 columns: divides shapes 256 does not (3584 = 16 x 224) and fills the pairs'
    // rounds there (3584^2: 224 tiles = 2.95 rounds of 76 pairs instead of 196 = 2.58
    // rounded up to 3 full-width rounds).  It is feasible on few swept shapes, so its
    // constants are the 256-wide tile's with the k-tile cost scaled by 0.96 (measured
    // at 3584^3 and 7168^3: the MMA time does not shrink in proportion to N) and the
    // streaming term by its operand bytes, 480 / 512.
    SDT_PAIR(224, 6, "2cta_256x224", 11.060, 0.21877, 0.000, 0.09862, true),
    // Skinny tiles for few-row problems (M up to a few tens, e.g. decode rows): the
    // operands are swapped so that the many output columns fill the 128 MMA rows and
    // the M rows become a 16- or 32-wide MMA N; the weights stream through a deep ring
    // (18 / 20 KB per stage) and C is written transposed back.  gemm_ex and
    // gemm_ex_splitk only; A must be stored M x K (K contiguous).
    SDT_STILE(16, 12, "s128x16", 7.0, 0.25),
    SDT_STILE(32, 11, "s128x32", 7.0, 0.25),
};
static constexpr int kNumTiles = sizeof(kLadder) / sizeof(kLadder[0]);
static_assert(sizeof(kSplitLaunch) / sizeof(kSplitLaunch[0]) == kNumTiles, "one split-K row per ladder tile");
static_assert(sizeof(kStreamLaunch) / sizeof(kStreamLaunch[0]) == kNumTiles, "one stream-K row per ladder tile");
static constexpr int kDefaultSmemLimit = 232448;  // opt-in shared memory per block on sm_100-class parts
static constexpr int kMaxRing = 24;
static constexpr int64_t kMaxDim = int64_t(1) << 30;
static constexpr int64_t kMaxGridTiles = 0x3fffffff;  // output tiles of one launch

// Ring depth of a launch: `req` when in 2..kMaxRing, else SDT_STAGES when set, else
// the tile's own depth; lowered until the ring fits in shared memory.
static int tile_stages(const LadderTile &t, int smem_limit, int req = 0) {
    int s = t.stages;
    if (req >= 2 && req <= kMaxRing) {
        s = req;
    } else if (const char *e = getenv("SDT_STAGES")) {
        int v = atoi(e);
        if (v >= 2 && v <= kMaxRing) s = v;
    }
    while (s > 2 && t.smem_fixed + s * t.smem_per_stage > smem_limit) --s;
    return s;
}

static int tile_smem(const LadderTile &t, int stages) { return t.smem_fixed + stages * t.smem_per_stage; }

static bool feasible(const LadderTile &t, int64_t M, int64_t N, int64_t K, int smem_limit) {
    if (t.swap) return false;  // gemm_ex forms only
    if (M <= 0 || N <= 0 || K <= 0) return false;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return false;
    if (M % t.BM || N % t.BN || K % kBK) return false;               // (i) divides the shape
    if (K / kBK < 2) return false;                                   // (ii) fills the pipeline
    if (tile_smem(t, t.stages) > smem_limit) return false;           // (iii) fits in shared memory
    if (t.tmem_cols > 512) return false;                             //       and in tensor memory
    return true;
}

static int ctas_per_sm(const LadderTile &t, int smem_per_sm) {
    int by_smem = smem_per_sm / (tile_smem(t, t.stages) + 1024);
    int by_tmem = 512 / t.tmem_cols;
    int by_threads = 2048 / t.threads;
    int occ = by_smem < by_tmem ? by_smem : by_tmem;
    occ = occ < by_threads ? occ : by_threads;
    return occ < 1 ? 1 : occ;
}

// Estimated run time (us) of `ctas` CTAs of non-persistent tile t, each walking
// `kpc` k-tiles: whole waves of co-resident CTAs, a round cost per wave.
static double wave_model_us(const LadderTile &t, double ctas, double kpc, int sm_count, int smem_per_sm) {
    const int occ = ctas_per_sm(t, smem_per_sm);
    const double per_wave = double(sm_count) * occ;
    const double waves = std::ceil(ctas / per_wave);
    // CTAs beyond the first on the busiest SM: occ - 1 in each full wave, and in the
    // last wave as many as its CTAs need
    const double full = std::floor(ctas / per_wave), rest = ctas - full * per_wave;
    double extra = full * (occ - 1);
    if (rest > 0) extra += std::min(double(occ), std::ceil(rest / sm_count)) - 1;
    return t.fixed_us + waves * (t.round_us + std::max(0.0, kpc - t.stages) * t.kt_us) +
           ctas * kpc / per_wave * t.bw_us + extra * t.share_us;
}

// Estimated run time (us) of tile t on the shape.  Persistent tiles: one worker
// (CTA or CTA pair) per SM (pair of SMs) walking ceil(tiles / workers) tiles.
// Other tiles: whole waves of co-resident CTAs.
static double model_us(const LadderTile &t, int64_t M, int64_t N, int64_t K, int sm_count, int smem_per_sm) {
    const double tiles = double((M + t.BM - 1) / t.BM) * double((N + t.BN - 1) / t.BN);
    const double nK = double((K + kBK - 1) / kBK);
    if (!t.persistent) return wave_model_us(t, tiles, nK, sm_count, smem_per_sm);
    const double workers = t.cta_group == 2 ? double(sm_count / 2) : double(sm_count);
    double rounds = std::ceil(tiles / workers);
    if (t.cta_group == 2 && t.BN == 256 && tiles >= workers) {
        // a tail of at most half the workers runs as half-width items in half a round
        // (after at least one full round: a grid that is all tail keeps the full
        // k-loop per item, which the fit does not cover)
        const double tail = tiles - std::floor(tiles / workers) * workers;
        if (tail > 0 && 2 * tail <= workers) rounds -= 0.5;
    }
    return t.fixed_us + std::max(0.0, rounds * nK - t.stages) * t.kt_us + rounds * t.round_us +
           tiles * nK / workers * t.bw_us;
}

static int pick_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit, int smem_per_sm) {
    int best = -1, fallback = -1;
    double best_cost = 0.0;
    for (int i = 0; i < kNumTiles; ++i) {
        if (!feasible(kLadder[i], M, N, K, smem_limit)) continue;
        if (fallback < 0) fallback = i;
        if (!kLadder[i].candidate) continue;
        const double c = model_us(kLadder[i], M, N, K, sm_count, smem_per_sm);
        if (best < 0 || c < best_cost * (1.0 - 1e-9)) {
            best = i;
            best_cost = c;
        }
    }
    return best >= 0 ? best : fallback;
}

// Tiles usable on any shape (they overhang ragged edges): only the on-chip limits apply.
static bool fits_chip(const LadderTile &t, int smem_limit) {
    return tile_smem(t, t.stages) <= smem_limit && t.tmem_cols <= 512;
}

static int pick_any(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit, int smem_per_sm) {
    int best = -1;
    double best_cost = 0.0;
    for (int i = 0; i < kNumTiles; ++i) {
        if (!kLadder[i].candidate || !fits_chip(kLadder[i], smem_limit)) continue;
        const double c = model_us(kLadder[i], M, N, K, sm_count, smem_per_sm);
        if (best < 0 || c < best_cost * (1.0 - 1e-9)) {
            best = i;
            best_cost = c;
        }
    }
    return best;
}

static int find_tile(const char *name) {
    for (int i = 0; i < kNumTiles; ++i)
        if (!strcmp(kLadder[i].name, name)) return i;
    return -1;
}

static bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

// ---- frozen tune table ------------------------------------------------------

struct TuneEntry {
    int tile;
    int stagger;  // -1 = auto
    int raster;   // m-tiles per raster band, 0 = default
    int stages;   // ring depth, 0 = the tile's own
};
using ShapeKey = std::tuple<int64_t, int64_t, int64_t>;
static std::mutex g_table_mu;
static std::map<ShapeKey, TuneEntry> g_table;
static std::once_flag g_env_table_once;

static int load_table_file(const char *path, std::map<ShapeKey, TuneEntry> *out) {
    FILE *f = fopen(path, "r");
    if (!f) return fail(SDT_ERR_TABLE, "cannot open tune table '%s'", path);
    char line[512];
    int lineno = 0;
    std::map<ShapeKey, TuneEntry> tab;
    while (fgets(line, sizeof line, f)) {
        ++lineno;
        char *hash = strchr(line, '#');
        if (!strchr(line, '\n') && !feof(f)) {
            // a line longer than the buffer: its rest is read and dropped, which is
            // only right when the cut falls inside a comment
            int c;
            while ((c = fgetc(f)) != EOF && c != '\n') {
            }
            if (!hash) {
                fclose(f);
                return fail(SDT_ERR_TABLE, "%s:%d: entry longer than %d characters", path, lineno,
                            int(sizeof line) - 2);
            }
        }
        if (hash) *hash = 0;
        long long M, N, K;
        char name[64];
        int stagger = -1, raster = 0, stages = 0;
        int n = sscanf(line, "%lld %lld %lld %63s %d %d %d", &M, &N, &K, name, &stagger, &raster, &stages);
        if (n <= 0) {
            bool blank = true;
            for (char *c = line; *c; ++c)
                if (*c != ' ' && *c != '\t' && *c != '\n' && *c != '\r') blank = false;
            if (blank) continue;
        }
        if (n < 4) {
            fclose(f);
            return fail(SDT_ERR_TABLE, "%s:%d: expected 'M N K tile [stagger [raster [stages]]]'", path, lineno);
        }
        int id = find_tile(name);
        if (id < 0) {
            fclose(f);
            return fail(SDT_ERR_TABLE, "%s:%d: unknown tile '%s'", path, lineno, name);
        }
        if (!feasible(kLadder[id], M, N, K, kDefaultSmemLimit)) {
            fclose(f);
            return fail(SDT_ERR_TABLE, "%s:%d: tile %s is infeasible for %lldx%lldx%lld", path, lineno, name,
                        M, N, K);
        }
        if (n >= 5 && stagger != 0 && stagger != 1 && stagger != -1) {
            fclose(f);
            return fail(SDT_ERR_TABLE, "%s:%d: stagger must be -1, 0 or 1", path, lineno);
        }
        if (n >= 6 && (raster < 0 || raster > (1 << 20))) {
            fclose(f);
            return fail(SDT_ERR_TABLE, "%s:%d: raster must be 0 (default) or a positive band height", path, lineno);
        }
        if (n >= 7 && stages != 0 && (stages < 2 || stages > kMaxRing)) {
            fclose(f);
            return fail(SDT_ERR_TABLE, "%s:%d: stages must be 0 (the tile's own) or 2..%d", path, lineno, kMaxRing);
        }
        tab[ShapeKey(M, N, K)] = TuneEntry{id, n >= 5 ? stagger : -1, n >= 6 ? raster : 0, n >= 7 ? stages : 0};
    }
    fclose(f);
    *out = std::move(tab);
    return SDT_OK;
}

static void load_env_table() {
    std::call_once(g_env_table_once, [] {
        const char *p = getenv("SDT_TUNE_TABLE");
        if (!p || !*p) return;
        std::map<ShapeKey, TuneEntry> tab;
        if (load_table_file(p, &tab) == SDT_OK) {
            std::lock_guard<std::mutex> lock(g_table_mu);
            g_table = std::move(tab);
        } else {
            fprintf(stderr, "libsdt: SDT_TUNE_TABLE ignored: %s\n", sdt_last_error());
        }
    });
}

static bool table_lookup(int64_t M, int64_t N, int64_t K, TuneEntry *e) {
    std::lock_guard<std::mutex> lock(g_table_mu);
    auto it = g_table.find(ShapeKey(M, N, K));
    if (it == g_table.end()) return false;
    *e = it->second;
    return true;
}

// ---- TMA tensor maps ---------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Cache key of one 2-D tensor map.  The row stride is part of the key: two
// operands of one shape but different pitch must never share a map.  The same
// function builds the key for the lookup and for the insert.
struct MapKey {
    uintptr_t ptr;
    uint64_t inner, outer, row_stride_bytes;
    int dtype, box_outer, box_inner, swizzle;
    bool operator<(const MapKey &o) const {
        return std::tie(ptr, inner, outer, row_stride_bytes, dtype, box_outer, box_inner, swizzle) <
               std::tie(o.ptr, o.inner, o.outer, o.row_stride_bytes, o.dtype, o.box_outer, o.box_inner, o.swizzle);
    }
};

static MapKey map_key(const void *ptr, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes, int dtype,
                      int box_outer, int box_inner, int swizzle) {
    return MapKey{reinterpret_cast<uintptr_t>(ptr), inner, outer, row_stride_bytes, dtype, box_outer, box_inner,
                  swizzle};
}

static std::mutex g_map_mu;
static std::map<MapKey, CUtensorMap> g_maps;
static uint64_t g_map_encodes = 0;

// 2-D 16-bit tensor map (fp16 or bf16) with a box of `box_inner` contiguous elements
// by `box_outer` rows; `inner` is the contiguous dimension.  Operand maps use 64 x
// rows boxes with the 128-byte swizzle: elements outside [0, inner) x [0, outer) read
// as zero, which is what lets tiles overhang ragged edges.  The C map of the TMA
// stores uses 32 x 32 boxes with the 64-byte swizzle: elements outside are not written.
static int tensor_map_2d(const void *ptr, int dtype, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                         int box_outer, CUtensorMap *out, int box_inner = 64,
                         CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    const MapKey key = map_key(ptr, inner, outer, row_stride_bytes, dtype, box_outer, box_inner, int(swizzle));
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return SDT_OK;
        }
    }
    auto fn = encode_fn();
    if (!fn) return fail(SDT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    CUtensorMap m;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        dtype == SDT_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(&m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SDT_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_maps.size() >= 4096) g_maps.clear();
    g_maps[key] = m;
    ++g_map_encodes;
    *out = m;
    return SDT_OK;
}

// Operand maps for the layouts: A is M x K (K contiguous) or, transposed, K x M;
// B is K x N (N contiguous) or, transposed, N x K.  A row-major A tile is one box
// of a_rows (the rows one CTA stages) x 64; every other operand tile is loaded as
// 64 x 64 boxes.
// Rows of a K-major B box: the tile width for narrow tiles, 64 for the rest, and a
// two-CTA tile's whole half width when that is not a multiple of 64 (256x224: 112).
static int b_box_rows(const LadderTile &t) {
    if (t.BN < 64) return t.BN;
    if (t.cta_group == 2 && (t.BN / 2) % 64) return t.BN / 2;
    return 64;
}

static int operand_maps(const void *A, int64_t lda, const void *B, int64_t ldb, int64_t M, int64_t N, int64_t K,
                        int dtype, int layout, int a_rows, CUtensorMap *tmA, CUtensorMap *tmB, int b_rows = 64) {
    const bool a_t = layout & SDT_LAYOUT_A_T, b_t = layout & SDT_LAYOUT_B_T;
    int rc = a_t ? tensor_map_2d(A, dtype, uint64_t(M), uint64_t(K), uint64_t(lda) * 2, 64, tmA)
                 : tensor_map_2d(A, dtype, uint64_t(K), uint64_t(M), uint64_t(lda) * 2, a_rows, tmA);
    if (rc) return rc;
    return b_t ? tensor_map_2d(B, dtype, uint64_t(K), uint64_t(N), uint64_t(ldb) * 2, b_rows, tmB)
               : tensor_map_2d(B, dtype, uint64_t(N), uint64_t(K), uint64_t(ldb) * 2, 64, tmB);
}

// A gemm_ex problem as the kernels see it.  Skinny (swap) tiles compute
// C^T = op(B)^T . op(A)^T: the new A is op(B)^T (stored as B is, with the
// transposed bit flipped), the new B is op(A)^T (A stored M x K becomes a
// K-contiguous [M][K] operand of N = M columns), and C is written transposed.
struct ExProblem {
    int64_t M, N, K;
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    int layout;
    int c_trans;
};

static int ex_problem(const LadderTile &t, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                      const void *B, int64_t ldb, int layout, ExProblem *out) {
    if (!t.swap) {
        *out = ExProblem{M, N, K, A, lda, B, ldb, layout, 0};
        return SDT_OK;
    }
    if (layout & SDT_LAYOUT_A_T)
        return fail(SDT_ERR_TILE, "skinny tile %s needs A stored M x K (K contiguous)", t.name);
    const int new_layout = ((layout & SDT_LAYOUT_B_T) ? 0 : SDT_LAYOUT_A_T) | SDT_LAYOUT_B_T;
    *out = ExProblem{N, M, K, B, ldb, A, lda, new_layout, 1};
    return SDT_OK;
}

// Instruction-descriptor bits for the types and majors: fp32 accumulator (bit 4),
// A/B type f16 = 0 / bf16 = 1 (bits 7 and 10), A MN-major (bit 15), B MN-major (bit 16).
static uint32_t idesc_flags_for(int dtype, int layout) {
    const uint32_t dt = dtype == SDT_DTYPE_BF16 ? 1u : 0u;
    const uint32_t a_mn = (layout & SDT_LAYOUT_A_T) ? 1u : 0u;
    const uint32_t b_mn = (layout & SDT_LAYOUT_B_T) ? 0u : 1u;
    return (1u << 4) | (dt << 7) | (dt << 10) | (a_mn << 15) | (b_mn << 16);
}

// ---- launch ----------------------------------------------------------------------

__global__ void splitk_reduce_kernel(const float *__restrict__ partials, uint16_t *__restrict__ C, int64_t M,
                                     int64_t N, int64_t Mp, int64_t Np, int64_t ldc, int splits, int bf16) {
    const int64_t vecs = N / 8, total = M * vecs, plane = Mp * Np;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = i / vecs, c = (i % vecs) * 8;
        const float *src = partials + r * Np + c;
        float4 a0 = __ldg(reinterpret_cast<const float4 *>(src));
        float4 a1 = __ldg(reinterpret_cast<const float4 *>(src + 4));
        for (int sp = 1; sp < splits; ++sp) {
            const float4 b0 = __ldg(reinterpret_cast<const float4 *>(src + sp * plane));
            const float4 b1 = __ldg(reinterpret_cast<const float4 *>(src + sp * plane + 4));
            a0.x += b0.x; a0.y += b0.y; a0.z += b0.z; a0.w += b0.w;
            a1.x += b1.x; a1.y += b1.y; a1.z += b1.z; a1.w += b1.w;
        }
        *reinterpret_cast<uint4 *>(C + r * ldc + c) = pack8_f32(a0, a1, bf16 != 0);
    }
}

__global__ void splitk_reduce_trans_kernel(const float *__restrict__ partials, uint16_t *__restrict__ C,
                                           int64_t M, int64_t N, int64_t Mp, int64_t Np, int64_t ldc, int splits,
                                           int bf16) {
    const int64_t total = M * N, plane = Mp * Np;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = i % M, c = i / M;
        const float *src = partials + r * Np + c;
        float a = src[0];
        for (int sp = 1; sp < splits; ++sp) a += src[sp * plane];
        C[c * ldc + r] = f32_to_16(a, bf16 != 0);
    }
}

__global__ void zero_fill_u32(unsigned *p, size_t n) {
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        p[i] = 0u;
}

// C[r][0..N) = 0 for r < M with row stride ldc (N, ldc multiples of 8).
__global__ void zero_fill_2d(uint16_t *C, int64_t M, int64_t N, int64_t ldc) {
    const int64_t vecs = N / 8, total = M * vecs;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x)
        *reinterpret_cast<uint4 *>(C + (i / vecs) * ldc + (i % vecs) * 8) = make_uint4(0, 0, 0, 0);
}

__global__ void zero_fill_f16(__half *C, size_t n) {
    size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x;
    const size_t stride = size_t(gridDim.x) * blockDim.x;
    for (; i < n; i += stride) C[i] = __ushort_as_half(0);
}

// A numeric knob: unset, empty or not a whole decimal number -> the default; else
// clamped to [lo, hi].
static int env_int(const char *name, int dflt, int lo, int hi) {
    const char *s = getenv(name);
    if (!s || !*s) return dflt;
    char *end = nullptr;
    errno = 0;
    const long v = strtol(s, &end, 10);
    if (end == s || *end != '\0' || errno == ERANGE) return dflt;
    return v < lo ? lo : (v > hi ? hi : int(v));
}

// SDT_STAGGER: "0"/"off", "1"/"on", or "auto" (default): on for the one-CTA tiles,
// off for the persistent and two-CTA kernels.  Those keep a whole grid of tiles in
// flight on the same k-slices, which L2 then serves once; staggering their k-loops
// measured 3-5 % slower on GB300 at 2048^3 and 4096^3 and no faster at 8192^3 and
// 12288^3 (alternating processes on one GPU); on the one-CTA tiles it is neutral.
static int stagger_default(const LadderTile &t) {
    const char *s = getenv("SDT_STAGGER");
    if (s && (!strcmp(s, "0") || !strcasecmp(s, "off"))) return 0;
    if (s && (!strcmp(s, "1") || !strcasecmp(s, "on"))) return 1;
    return t.persistent ? 0 : 1;
}

static int validate_common(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C) {
    if (M < 0 || N < 0 || K < 0) return fail(SDT_ERR_SHAPE, "negative dimension (M=%lld N=%lld K=%lld)",
                                             (long long)M, (long long)N, (long long)K);
    if (M == 0 || N == 0) return SDT_OK;
    if (!C || (K > 0 && (!A || !B))) return fail(SDT_ERR_NULL, "NULL operand pointer");
    if ((reinterpret_cast<uintptr_t>(C) & 15) || (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15) ||
                                                             (reinterpret_cast<uintptr_t>(B) & 15))))
        return fail(SDT_ERR_ALIGN, "A, B and C must be 16-byte aligned");
    return SDT_OK;
}

// Workspaces of the split-K family and of the two-CTA tail begin with a fixed 1 MiB
// region of u32 arrival counters; the fp32 partials follow it.
static constexpr size_t kCounterRegionBytes = size_t(1) << 20;

// ---- the last round of the two-CTA kernel -----------------------------------------
//
// T tiles on P pairs leave L = T mod P tiles (all T when T < P) for a last round in
// which P - L pairs idle.  That round runs in one of three forms:
//   whole   the L tiles as they are;
//   halves  two half-width items per tile (BN = 256 and 2L <= P);
//   k-split given a workspace, S full-width items per tile over consecutive k-ranges
//           (L*S <= P) whose fp32 partials the last to finish sums.  Split 0 is made
//           longer than the others by the time a partial takes to be published, so
//           that it normally finishes last and sums without publishing its own.
// The estimate of each form's last round uses GB300 timings of the 256 x 256 pair
// kernel at 4096^3 (globaltimer stamps, cold L2): a k-tile of the last round takes
// 0.297 us in whole-width items, 0.272 us in half-width ones and 0.366 us in k-split
// items (their partials' traffic shares L2 with the operand loads); from the last MMA
// issue to the stores' completion 2.4 us for a plain epilogue; for the summing split
// 4.1 us with two splits (it watched the other split's count during its last k-tiles
// and read the other partial straight from L2) or 9.7 us + 2.5 us per split beyond
// two (it copies the others through shared memory).  Split 0 leads the others by 12
// k-tiles, the time a partial takes to be published.  So at 4096^3 two k-ranges
// (39 x 0.366 + 4.1 = 18.4 us) beat half-width items (64 x 0.272 + 2.4 = 19.8 us), at
// 2560^3 they do not (13.6 against 13.3 us).
// The cheapest form is planned; `req` forces the k-split count (>= 2) or disables it (0).
struct PairTail {
    int tail_start, num_items, splits, long_k;
};

static constexpr int kPairTailMaxSplits = 8;
static constexpr double kTailKt = 0.297, kTailHalfKt = 0.272, kTailSplitKt = 0.366, kTailEpi = 2.4,
                        kTailReduce2 = 4.1, kTailReduceN = 9.7, kTailReduceExtra = 2.5;
static constexpr int kTailLead = 12;  // k-tiles by which split 0 outlasts the others

// The largest k-split count for L leftover tiles: L*S <= P, S <= nK, and the other
// S-1 partials of a 64-column group must fit in an epilogue warp's quarter of the ring.
static int pair_tail_max_splits(const LadderTile &t, int leftover, int pairs, int nK, int stages) {
    if (leftover <= 0) return 1;
    const int quarter = (stages * t.smem_per_stage / 4) & ~1023;
    int s = std::min(std::min(pairs / leftover, nK), kPairTailMaxSplits);
    while (s > 1 && (s - 1) * 64 * 32 * 4 > quarter) --s;
    return std::max(s, 1);
}

// k-tiles of split 0 for an S-way split of nK k-tiles: the others' share plus the
// lead, at most nK - (S-1) (every other split keeps at least one k-tile).
static int pair_tail_long(int nK, int S) {
    const int want = (nK + (S - 1) * kTailLead + S - 1) / S;
    return std::max(std::min(want, nK - (S - 1)), (nK + S - 1) / S);
}

static PairTail pair_tail_plan(const LadderTile &t, int tiles, int nK, int pairs, int stages, bool have_ws,
                               int req) {
    PairTail pt{tiles, tiles, 0, 0};
    if (t.cta_group != 2 || pairs <= 0 || tiles <= 0) return pt;
    const int L = tiles % pairs;
    if (L == 0) return pt;
    double best = nK * kTailKt + kTailEpi;  // whole tiles
    int form = 0;                           // 0 whole, 1 halves, >= 2 k-split count
    if (t.BN == 256 && 2 * L <= pairs && env_int("SDT_TAIL_SPLIT", 1, 0, 1) && nK * kTailHalfKt + kTailEpi < best) {
        best = nK * kTailHalfKt + kTailEpi;
        form = 1;
    }
    const int smax = have_ws ? pair_tail_max_splits(t, L, pairs, nK, stages) : 1;
    if (req >= 2 && smax >= 2) {
        form = std::min(req, smax);
    } else if (req != 0) {
        for (int sp = 2; sp <= smax; ++sp) {
            const double c = pair_tail_long(nK, sp) * kTailSplitKt +
                             (sp == 2 ? kTailReduce2 : kTailReduceN + kTailReduceExtra * (sp - 2));
            if (c < best) {
                best = c;
                form = sp;
            }
        }
    }
    pt.tail_start = tiles - L;
    if (form == 1) {
        pt.num_items = pt.tail_start + 2 * L;
    } else if (form >= 2) {
        pt.num_items = pt.tail_start + L * form;
        pt.splits = form;
        pt.long_k = pair_tail_long(nK, form);
    } else {
        pt.tail_start = tiles;
    }
    return pt;
}

// Workspace bytes a two-CTA launch with k-split tail items needs: the counter region
// and one 256 x BN fp32 slot per item.
static size_t pair_tail_ws_bytes(const LadderTile &t, int items) {
    return kCounterRegionBytes + size_t(items) * 256 * size_t(t.BN) * 4;
}

// A caller workspace for the two-CTA tail (gemm_f16_ws / gemm_ex_ws); ws == nullptr
// means none.  req: -1 plan the tail, 0 no k-split, >= 2 this k-split count.
struct TailWs {
    void *ws;
    size_t bytes;
    int req;
};

// Launches ladder tile `tile_id` on validated, non-empty arguments with K > 0
// (any shape: tiles overhang ragged edges; layouts and type per the flags).
static int run_tile_ex(int tile_id, int stagger_req, int64_t M0, int64_t N0, int64_t K0, const void *A0,
                       int64_t lda0, const void *B0, int64_t ldb0, void *C, int64_t ldc, int dtype, int layout0,
                       cudaStream_t stream, const DeviceInfo &dev, int raster_req = 0, int stages_req = 0,
                       const TailWs *tw = nullptr) {
    const LadderTile &t = kLadder[tile_id];
    ExProblem ex;
    int rc = ex_problem(t, M0, N0, K0, A0, lda0, B0, ldb0, layout0, &ex);
    if (rc) return rc;
    const int64_t M = ex.M, N = ex.N, K = ex.K, lda = ex.lda, ldb = ex.ldb;
    const void *A = ex.A, *B = ex.B;
    const int layout = ex.layout;
    CUtensorMap tmA, tmB;
    rc = operand_maps(A, lda, B, ldb, M, N, K, dtype, layout, t.BM / t.cta_group, &tmA, &tmB, b_box_rows(t));
    if (rc) return rc;
    int *status = nullptr;
    rc = status_word(&status);
    if (rc) return rc;

    GemmArgs a;
    memset(&a, 0, sizeof a);
    a.C = static_cast<__half *>(C);
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.num_m_tiles = int((M + t.BM - 1) / t.BM);
    a.num_n_tiles = int((N + t.BN - 1) / t.BN);
    a.num_k_tiles = int((K + kBK - 1) / kBK);
    a.stages = tile_stages(t, dev.smem_optin, stages_req);
    const int want_stagger = stagger_req < 0 ? stagger_default(t) : stagger_req;
    a.stagger = (want_stagger && is_pow2(a.num_k_tiles)) ? 1 : 0;
    a.stagger_stride = env_int("SDT_STAGGER_STRIDE", 1, 1, 1 << 20);
    a.raster_group = raster_req > 0 ? raster_req : env_int("SDT_RASTER_GROUP", 8, 1, 1 << 20);
    a.timeout_ns = wait_timeout_ns();
    a.status = status;
    a.max_ctas = dev.sm_count * ctas_per_sm(t, dev.smem_per_sm);
    a.ldc = int(ldc);
    a.idesc_flags = idesc_flags_for(dtype, layout);
    a.c_trans = ex.c_trans;
    if (int64_t(a.num_m_tiles) * a.num_n_tiles > kMaxGridTiles)
        return fail(SDT_ERR_SHAPE, "grid too large");
    const int tiles = a.num_m_tiles * a.num_n_tiles;
    const bool have_ws = tw && tw->ws;
    int tail_req = have_ws ? tw->req : 0;
    if (have_ws && tail_req < 0) tail_req = env_int("SDT_TAIL_KSPLIT", -1, -1, kPairTailMaxSplits);
    const PairTail pt = pair_tail_plan(t, tiles, a.num_k_tiles, std::max(1, a.max_ctas / 2), a.stages, have_ws,
                                       tail_req);
    a.tail_start = pt.tail_start;
    a.num_items = pt.num_items;
    a.tail_splits = pt.splits;
    a.tail_long = pt.long_k;
    if (pt.splits >= 2) {
        if (pair_tail_ws_bytes(t, pt.num_items - pt.tail_start) > tw->bytes)
            return fail(SDT_ERR_ARG, "workspace of %zu bytes is too small for the two-CTA tail (%zu)", tw->bytes,
                        pair_tail_ws_bytes(t, pt.num_items - pt.tail_start));
        a.counters = static_cast<unsigned *>(tw->ws);
        a.partials = reinterpret_cast<float *>(static_cast<char *>(tw->ws) + kCounterRegionBytes);
    }
    // the persistent and two-CTA kernels write C with TMA stores (32 x 32 boxes)
    CUtensorMap tmC = tmA;  // unused by the one-CTA kernel
    if (t.persistent) {
        rc = tensor_map_2d(C, dtype, uint64_t(N), uint64_t(M), uint64_t(ldc) * 2, 32, &tmC, 32,
                           CU_TENSOR_MAP_SWIZZLE_64B);
        if (rc) return rc;
    }
    int e = t.launch[layout & 3](tmA, tmB, tmC, a, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SDT_ERR_LAUNCH, "launch of tile %s failed: %s", t.name, cudaGetErrorString(cudaError_t(e)));
    }
    return SDT_OK;
}

// gemm_f16's forced tile: tight row-major fp16, the tile must divide the shape.
static int run_tile(int tile_id, int stagger_req, int64_t M, int64_t N, int64_t K, const void *A,
                    const void *B, void *C, cudaStream_t stream, const DeviceInfo &dev, int raster_req = 0,
                    int stages_req = 0, const TailWs *tw = nullptr) {
    const LadderTile &t = kLadder[tile_id];
    if (!feasible(t, M, N, K, dev.smem_optin))
        return fail(SDT_ERR_TILE, "tile %s is infeasible for %lldx%lldx%lld", t.name, (long long)M,
                    (long long)N, (long long)K);
    return run_tile_ex(tile_id, stagger_req, M, N, K, A, K, B, N, C, N, SDT_DTYPE_F16, 0, stream, dev, raster_req,
                       stages_req, tw);
}

// SDT_AUTOTUNE=1: time every feasible tile on the caller's stream (synchronising
// it) and remember the fastest for this shape.
static int autotune_shape(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                          cudaStream_t stream, const DeviceInfo &dev, TuneEntry *out) {
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) {
        cudaGetLastError();
        return fail(SDT_ERR_CUDA, "cudaEventCreate failed during autotune");
    }
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaGetLastError();
        cudaEventDestroy(e0);
        return fail(SDT_ERR_CUDA, "cudaEventCreate failed during autotune");
    }
    int best = -1;
    float best_ms = 0.f;
    for (int i = 0; i < kNumTiles; ++i) {
        if (!feasible(kLadder[i], M, N, K, dev.smem_optin)) continue;
        int rc = run_tile(i, -1, M, N, K, A, B, C, stream, dev);
        if (rc) {  // the launch error of this tile, not a later "nothing feasible"
            cudaEventDestroy(e0);
            cudaEventDestroy(e1);
            return rc;
        }
        cudaEventRecord(e0, stream);
        for (int r = 0; r < 5 && rc == SDT_OK; ++r) rc = run_tile(i, -1, M, N, K, A, B, C, stream, dev);
        cudaEventRecord(e1, stream);
        if (cudaEventSynchronize(e1) != cudaSuccess) {
            cudaGetLastError();
            rc = fail(SDT_ERR_CUDA, "autotune timing failed");
        }
        if (rc) {
            cudaEventDestroy(e0);
            cudaEventDestroy(e1);
            return rc;
        }
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        if (best < 0 || ms < best_ms) {
            best = i;
            best_ms = ms;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (best < 0) return fail(SDT_ERR_SHAPE, "no feasible tile to autotune");
    *out = TuneEntry{best, -1, 0, 0};
    std::lock_guard<std::mutex> lock(g_table_mu);
    g_table[ShapeKey(M, N, K)] = *out;
    return SDT_OK;
}

static int gemm_dispatch(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                         sdt_stream_t stream_h, int tile_id, int stagger, const TailWs *tw = nullptr) {
    clear_error();
    int rc = validate_common(M, N, K, A, B, C);
    if (rc) return rc;
    if (M == 0 || N == 0) return SDT_OK;
    if (stagger < -1 || stagger > 1) return fail(SDT_ERR_ARG, "stagger must be -1, 0 or 1");
    if (tile_id != -1 && (tile_id < 0 || tile_id >= kNumTiles))
        return fail(SDT_ERR_TILE, "unknown tile id %d", tile_id);
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    if (K == 0) {
        if (M > kMaxDim || N > kMaxDim) return fail(SDT_ERR_SHAPE, "dimension too large");
        const size_t n = size_t(M) * size_t(N);
        const unsigned blocks = unsigned(std::min<size_t>((n + 255) / 256, size_t(dev.sm_count) * 8));
        zero_fill_f16<<<blocks, 256, 0, stream>>>(static_cast<__half *>(C), n);
        cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? SDT_OK : fail(SDT_ERR_LAUNCH, "zero fill failed: %s", cudaGetErrorString(e));
    }
    if (N % 8 || K % 8) return fail(SDT_ERR_SHAPE, "N and K must be multiples of 8");
    if (tile_id >= 0) return run_tile(tile_id, stagger, M, N, K, A, B, C, stream, dev, 0, 0, tw);

    load_env_table();
    TuneEntry te;
    if (table_lookup(M, N, K, &te) && feasible(kLadder[te.tile], M, N, K, dev.smem_optin))
        return run_tile(te.tile, stagger >= 0 ? stagger : te.stagger, M, N, K, A, B, C, stream, dev, te.raster,
                        te.stages, tw);
    if (env_flag("SDT_AUTOTUNE")) {
        rc = autotune_shape(M, N, K, A, B, C, stream, dev, &te);
        if (rc) return rc;
        return run_tile(te.tile, stagger, M, N, K, A, B, C, stream, dev, 0, 0, tw);
    }
    const int id = pick_for(M, N, K, dev.sm_count, dev.smem_optin, dev.smem_per_sm);
    if (id < 0)
        return fail(SDT_ERR_SHAPE, "no feasible tile for %lldx%lldx%lld (need M,N,K multiples of 64 and K >= 128)",
                    (long long)M, (long long)N, (long long)K);
    return run_tile(id, stagger, M, N, K, A, B, C, stream, dev, 0, 0, tw);
}

// ---- split-K ----------------------------------------------------------------------

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Workspace layout: a fixed 1 MiB region of u32 arrival counters (split-K in-kernel:
// one per output tile; stream-K: one per output tile and TMEM lane quarter), then the
// fp32 partials.  The counter region has the same place and size for every shape,
// tile, split count and algorithm: a completed call leaves its counters at zero and
// writes partials only past the region, so a workspace zeroed once serves any
// sequence of calls that do not overlap on the GPU.
static constexpr int64_t kMaxCounters = int64_t(kCounterRegionBytes / 4);
static size_t splitk_counter_bytes(int64_t) { return kCounterRegionBytes; }
static size_t splitk_partials_bytes(int64_t Mp, int64_t Np, int splits) {
    return size_t(splits) * size_t(Mp) * size_t(Np) * 4;
}

static int splitk_effective(int64_t nK, int splits) {
    const int64_t kps = ceil_div(nK, splits);
    return int(ceil_div(nK, kps));
}

static bool splitk_tile_ok(int tile_id) {
    return tile_id >= 0 && tile_id < kNumTiles && kSplitLaunch[tile_id][0] != nullptr;
}

// Dimensions the launches take (they refuse the rest); the size queries apply the same
// limits, so that their products stay far inside 64 bits.
static bool dims_in_range(int64_t M, int64_t N, int64_t K) {
    return M > 0 && N > 0 && K > 0 && M <= kMaxDim && N <= kMaxDim && K <= kMaxDim;
}

// Workspace bytes of split-K with tile t on any shape (0 for an invalid combination).
static size_t splitk_ws_bytes(const LadderTile &t, int64_t M, int64_t N, int64_t K, int splits) {
    if (!dims_in_range(M, N, K)) return 0;
    const int64_t nK = ceil_div(K, kBK);
    if (splits < 1 || splits > nK) return 0;
    const int64_t mt = ceil_div(M, t.BM), nt = ceil_div(N, t.BN);
    if (mt * nt > kMaxGridTiles) return 0;
    return splitk_counter_bytes(mt * nt) + splitk_partials_bytes(mt * t.BM, nt * t.BN, splitk_effective(nK, splits));
}

static bool splitk_feasible(const LadderTile &t, int64_t M, int64_t N, int64_t K, int smem_limit) {
    if (t.swap) return false;  // gemm_ex_splitk only
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return false;
    if (M % t.BM || N % t.BN || K % kBK) return false;
    return tile_smem(t, t.stages) <= smem_limit && t.tmem_cols <= 512;
}

// Cost model for (tile, splits): the tile model with K divided among the splits,
// CTAs = tiles x splits, plus the reduction's fp32 traffic (written once, read once).
static double splitk_model_us(const LadderTile &t, int64_t M, int64_t N, int64_t K, int splits, int sm_count,
                              int smem_per_sm) {
    const double ctas = double(ceil_div(M, t.BM)) * double(ceil_div(N, t.BN)) * splits;
    const double kps = double(ceil_div(ceil_div(K, kBK), splits));
    double us = wave_model_us(t, ctas, kps, sm_count, smem_per_sm);
    if (splits > 1) us += 1.0 + double(M) * double(N) * (8.0 * splits + 2.0) / 4.0e6;  // ~4 TB/s through L2
    return us;
}

static int pick_splitk_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit, int smem_per_sm,
                           int *tile_out, int *splits_out) {
    double best = 0.0;
    int bt = -1, bs = 1;
    const int64_t nK = K / kBK;
    for (int i = 0; i < kNumTiles; ++i) {
        if (!splitk_tile_ok(i) || !kLadder[i].candidate) continue;
        if (!splitk_feasible(kLadder[i], M, N, K, smem_limit)) continue;
        for (int sp = 1; sp <= 32 && sp <= nK; ++sp) {
            if (splitk_effective(nK, sp) != sp) continue;
            const double c = splitk_model_us(kLadder[i], M, N, K, sp, sm_count, smem_per_sm);
            if (bt < 0 || c < best * (1.0 - 1e-9)) {
                best = c;
                bt = i;
                bs = sp;
            }
        }
    }
    if (bt < 0) return fail(SDT_ERR_SHAPE, "no tile divides %lldx%lldx%lld", (long long)M, (long long)N, (long long)K);
    *tile_out = bt;
    *splits_out = bs;
    return SDT_OK;
}

// Launches split-K with tile `tile_id` (which has a split-K form and fits on chip)
// on validated, non-empty operands with K > 0; any shape (tiles overhang ragged
// edges: the TMA reads zeros outside the operands, the partial planes are whole
// tiles, the reduction writes only inside C), either layout bit, fp16 or bf16.
static int splitk_launch_ex(int tile_id, int splits, int algo, int64_t M0, int64_t N0, int64_t K0, const void *A0,
                            int64_t lda0, const void *B0, int64_t ldb0, void *C, int64_t ldc, int dtype, int layout0,
                            void *ws, size_t ws_bytes, cudaStream_t stream, const DeviceInfo &dev) {
    const LadderTile &t = kLadder[tile_id];
    ExProblem ex;
    int rc0 = ex_problem(t, M0, N0, K0, A0, lda0, B0, ldb0, layout0, &ex);
    if (rc0) return rc0;
    const int64_t M = ex.M, N = ex.N, K = ex.K, lda = ex.lda, ldb = ex.ldb;
    const void *A = ex.A, *B = ex.B;
    const int layout = ex.layout;
    const int64_t nK = ceil_div(K, kBK);
    if (splits < 1 || splits > nK) return fail(SDT_ERR_ARG, "splits must be in 1..%lld", (long long)nK);
    splits = splitk_effective(nK, splits);
    const int64_t mt = ceil_div(M, t.BM), nt = ceil_div(N, t.BN);
    if (mt * nt > kMaxGridTiles) return fail(SDT_ERR_SHAPE, "grid too large");
    if (algo == SDT_SPLITK_IN_KERNEL && mt * nt > kMaxCounters)
        return fail(SDT_ERR_SHAPE, "the in-kernel reduction counts at most %lld output tiles", (long long)kMaxCounters);
    const size_t need = splitk_ws_bytes(t, M, N, K, splits);
    if (!ws) return fail(SDT_ERR_NULL, "split-K needs a workspace");
    if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(SDT_ERR_ALIGN, "the workspace must be 256-byte aligned");
    if (ws_bytes < need)
        return fail(SDT_ERR_ARG, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes, need);
    CUtensorMap tmA, tmB;
    int rc = operand_maps(A, lda, B, ldb, M, N, K, dtype, layout, t.BM, &tmA, &tmB, t.BN < 64 ? t.BN : 64);
    if (rc) return rc;
    int *status = nullptr;
    rc = status_word(&status);
    if (rc) return rc;
    GemmArgs a;
    memset(&a, 0, sizeof a);
    a.ldc = int(ldc);
    a.idesc_flags = idesc_flags_for(dtype, layout);
    a.c_trans = ex.c_trans;
    a.C = static_cast<__half *>(C);
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.num_m_tiles = int(mt);
    a.num_n_tiles = int(nt);
    a.num_k_tiles = int(nK);
    a.stages = tile_stages(t, dev.smem_optin);
    a.stagger = 0;
    a.stagger_stride = 1;
    a.raster_group = env_int("SDT_RASTER_GROUP", 8, 1, 1 << 20);
    a.timeout_ns = wait_timeout_ns();
    a.status = status;
    a.max_ctas = dev.sm_count * ctas_per_sm(t, dev.smem_per_sm);
    a.splits = splits;
    a.k_per_split = int(ceil_div(nK, splits));
    a.splitk_reduce_in_kernel = algo == SDT_SPLITK_IN_KERNEL ? 1 : 0;
    a.counters = static_cast<unsigned *>(ws);
    a.partials = reinterpret_cast<float *>(static_cast<char *>(ws) + splitk_counter_bytes(mt * nt));
    int e = kSplitLaunch[tile_id][layout & 3](tmA, tmB, a, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SDT_ERR_LAUNCH, "split-K launch of tile %s failed: %s", t.name, cudaGetErrorString(cudaError_t(e)));
    }
    if (algo == SDT_SPLITK_REDUCE_KERNEL) {
        const int64_t total = ex.c_trans ? M * N : M * (N / 8);
        const unsigned blocks = unsigned(std::min<int64_t>((total + 255) / 256, int64_t(dev.sm_count) * 8));
        if (ex.c_trans)
            splitk_reduce_trans_kernel<<<blocks, 256, 0, stream>>>(a.partials, static_cast<uint16_t *>(C), M, N,
                                                                   mt * t.BM, nt * t.BN, ldc, splits,
                                                                   dtype == SDT_DTYPE_BF16 ? 1 : 0);
        else
            splitk_reduce_kernel<<<blocks, 256, 0, stream>>>(a.partials, static_cast<uint16_t *>(C), M, N, mt * t.BM,
                                                             nt * t.BN, ldc, splits, dtype == SDT_DTYPE_BF16 ? 1 : 0);
        cudaError_t e2 = cudaGetLastError();
        if (e2 != cudaSuccess) return fail(SDT_ERR_LAUNCH, "split-K reduction launch failed: %s", cudaGetErrorString(e2));
    }
    return SDT_OK;
}

// ---- stream-K ---------------------------------------------------------------------

// Tile index of output tile (m_tile, n_tile) in the banded raster order of
// tile_coords (bands of `group` m-tiles, m fastest within a band).
__device__ __forceinline__ int raster_index(int m_tile, int n_tile, int num_m, int num_n, int group) {
    const int band = m_tile / group;
    const int first_m = band * group;
    const int band_m = min(num_m - first_m, group);
    return band * group * num_n + n_tile * band_m + (m_tile - first_m);
}

// The separate fix-up of Stream-K: for every output tile that several CTAs share,
// sums their fp32 partial tiles in CTA order (the in-kernel fix-up's order) and
// writes C; tiles one CTA covered whole were stored by the GEMM kernel and are
// skipped.  One thread per 8 consecutive columns of a row of the problem as the
// kernel saw it (swapped for a skinny tile: c_trans writes C transposed).
__global__ void streamk_reduce_kernel(const float *__restrict__ partials, uint16_t *__restrict__ C, int M, int N,
                                      int64_t ldc, int BM, int BN, int num_m, int num_n, int nK, int G, int group,
                                      int c_trans, int bf16) {
    const int64_t chunks = (int64_t(N) + 7) / 8, total = int64_t(M) * chunks;
    const long long U = static_cast<long long>(num_m) * num_n * nK;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
        const int r = int(i / chunks), c0 = int(i % chunks) * 8;
        const int m_tile = r / BM, n_tile = c0 / BN;
        const int tile = raster_index(m_tile, n_tile, num_m, num_n, group);
        const long long u0 = static_cast<long long>(tile) * nK;
        const int g_lo = sk_owner(u0, G, U), g_hi = sk_owner(u0 + nK - 1, G, U);
        if (g_lo == g_hi) continue;  // whole tile, already in C
        const int lo_slot = 2 * g_lo + (sk_first_unit(g_lo, G, U) / nK == tile ? 0 : 1);
        const size_t off = size_t(r - m_tile * BM) * BN + (c0 - n_tile * BN);
        float v[8];
        {
            const float *src = partials + size_t(lo_slot) * BM * BN + off;
            const float4 a = __ldg(reinterpret_cast<const float4 *>(src)), b = __ldg(reinterpret_cast<const float4 *>(src + 4));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
        for (int g = g_lo + 1; g <= g_hi; ++g) {
            const float *src = partials + size_t(2 * g) * BM * BN + off;
            const float4 a = __ldg(reinterpret_cast<const float4 *>(src)), b = __ldg(reinterpret_cast<const float4 *>(src + 4));
            v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w; v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
        }
        if (c_trans) {
            for (int t = 0; t < 8; ++t)
                if (c0 + t < N) C[int64_t(c0 + t) * ldc + r] = f32_to_16(v[t], bf16 != 0);
        } else if (c0 + 8 <= N) {  // N % 8 == 0 unless swapped
            *reinterpret_cast<uint4 *>(C + int64_t(r) * ldc + c0) =
                pack8_f32(make_float4(v[0], v[1], v[2], v[3]), make_float4(v[4], v[5], v[6], v[7]), bf16 != 0);
        }
    }
}

static constexpr int64_t kMaxStreamUnits = int64_t(1) << 40;  // keeps (u + 1) * G within 64 bits
static constexpr int64_t kMaxStreamCtas = int64_t(1) << 20;

static bool streamk_tile_ok(int tile_id) {
    return tile_id >= 0 && tile_id < kNumTiles && kStreamLaunch[tile_id][0] != nullptr;
}

// CTAs of tile t's stream-K kernel that fit on one SM: shared memory at the ring depth
// the launch uses, two TMEM accumulators of BN columns, 192 threads.
static int streamk_ctas_per_sm(const LadderTile &t, int smem_limit, int smem_per_sm) {
    const int by_smem = smem_per_sm / (tile_smem(t, tile_stages(t, smem_limit)) + 1024);
    const int tmem = 2 * t.BN < 32 ? 32 : 2 * t.BN;
    int occ = std::min(by_smem, 512 / tmem);
    occ = std::min(occ, 2048 / 192);
    return occ < 1 ? 1 : occ;
}

// Workspace bytes of stream-K with tile t and `ctas` CTAs (lowered to the unit count)
// on an M x N x K problem as the kernel sees it (swapped for a skinny tile), 0 for an
// invalid combination: the counter region, then two fp32 BM x BN partial tiles per CTA.
static size_t streamk_ws_bytes(const LadderTile &t, int64_t M, int64_t N, int64_t K, int64_t ctas) {
    if (!dims_in_range(M, N, K) || ctas < 1 || ctas > kMaxStreamCtas) return 0;
    const int64_t tiles = ceil_div(M, t.BM) * ceil_div(N, t.BN);
    const int64_t units = tiles * ceil_div(K, kBK);
    if (4 * tiles > kMaxCounters || units > kMaxStreamUnits) return 0;
    return kCounterRegionBytes + size_t(2 * std::min(ctas, units)) * size_t(t.BM) * size_t(t.BN) * 4;
}

// Launches stream-K with tile `tile_id` (which has a stream-K form and fits on chip) on
// validated, non-empty operands with K > 0; ctas <= 0 takes one CTA per SM slot.  The
// CTA count is lowered to the number of (tile, k-tile) units when it is larger.
static int streamk_launch_ex(int tile_id, int64_t ctas, int algo, int64_t M0, int64_t N0, int64_t K0, const void *A0,
                             int64_t lda0, const void *B0, int64_t ldb0, void *C, int64_t ldc, int dtype, int layout0,
                             void *ws, size_t ws_bytes, cudaStream_t stream, const DeviceInfo &dev) {
    const LadderTile &t = kLadder[tile_id];
    ExProblem ex;
    int rc = ex_problem(t, M0, N0, K0, A0, lda0, B0, ldb0, layout0, &ex);
    if (rc) return rc;
    const int64_t M = ex.M, N = ex.N, K = ex.K;
    const int64_t nK = ceil_div(K, kBK);
    const int64_t mt = ceil_div(M, t.BM), nt = ceil_div(N, t.BN);
    if (4 * mt * nt > kMaxCounters)
        return fail(SDT_ERR_SHAPE, "stream-K counts at most %lld output tiles", (long long)(kMaxCounters / 4));
    const int64_t units = mt * nt * nK;
    if (units > kMaxStreamUnits) return fail(SDT_ERR_SHAPE, "too many (tile, k-tile) units for stream-K");
    if (ctas <= 0) ctas = int64_t(dev.sm_count) * streamk_ctas_per_sm(t, dev.smem_optin, dev.smem_per_sm);
    if (ctas > kMaxStreamCtas) return fail(SDT_ERR_ARG, "stream-K takes at most %lld CTAs", (long long)kMaxStreamCtas);
    ctas = std::min(ctas, units);
    const size_t need = streamk_ws_bytes(t, M, N, K, ctas);
    if (!ws) return fail(SDT_ERR_NULL, "stream-K needs a workspace");
    if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(SDT_ERR_ALIGN, "the workspace must be 256-byte aligned");
    if (ws_bytes < need)
        return fail(SDT_ERR_ARG, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes, need);
    CUtensorMap tmA, tmB;
    rc = operand_maps(ex.A, ex.lda, ex.B, ex.ldb, M, N, K, dtype, ex.layout, t.BM, &tmA, &tmB, t.BN < 64 ? t.BN : 64);
    if (rc) return rc;
    int *status = nullptr;
    rc = status_word(&status);
    if (rc) return rc;
    GemmArgs a;
    memset(&a, 0, sizeof a);
    a.ldc = int(ldc);
    a.idesc_flags = idesc_flags_for(dtype, ex.layout);
    a.c_trans = ex.c_trans;
    a.C = static_cast<__half *>(C);
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.num_m_tiles = int(mt);
    a.num_n_tiles = int(nt);
    a.num_k_tiles = int(nK);
    a.stages = tile_stages(t, dev.smem_optin);
    a.stagger_stride = 1;
    a.raster_group = env_int("SDT_RASTER_GROUP", 8, 1, 1 << 20);
    a.timeout_ns = wait_timeout_ns();
    a.status = status;
    a.max_ctas = int(ctas);
    a.splits = int(ctas);
    a.splitk_reduce_in_kernel = algo == SDT_SPLITK_STREAM ? 1 : 0;
    a.counters = static_cast<unsigned *>(ws);
    a.partials = reinterpret_cast<float *>(static_cast<char *>(ws) + kCounterRegionBytes);
    int e = kStreamLaunch[tile_id][ex.layout & 3](tmA, tmB, a, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SDT_ERR_LAUNCH, "stream-K launch of tile %s failed: %s", t.name, cudaGetErrorString(cudaError_t(e)));
    }
    if (algo == SDT_SPLITK_STREAM_REDUCE) {
        const int64_t total = M * ((N + 7) / 8);
        const unsigned blocks = unsigned(std::min<int64_t>((total + 255) / 256, int64_t(dev.sm_count) * 8));
        streamk_reduce_kernel<<<blocks, 256, 0, stream>>>(a.partials, static_cast<uint16_t *>(C), a.M, a.N, ldc, t.BM,
                                                          t.BN, a.num_m_tiles, a.num_n_tiles, a.num_k_tiles, a.splits,
                                                          a.raster_group, ex.c_trans, dtype == SDT_DTYPE_BF16 ? 1 : 0);
        cudaError_t e2 = cudaGetLastError();
        if (e2 != cudaSuccess) return fail(SDT_ERR_LAUNCH, "stream-K fix-up launch failed: %s", cudaGetErrorString(e2));
    }
    return SDT_OK;
}

static bool splitk_algo_ok(int algo) {
    return algo == SDT_SPLITK_REDUCE_KERNEL || algo == SDT_SPLITK_IN_KERNEL || algo == SDT_SPLITK_STREAM ||
           algo == SDT_SPLITK_STREAM_REDUCE;
}
static bool is_streamk(int algo) { return algo == SDT_SPLITK_STREAM || algo == SDT_SPLITK_STREAM_REDUCE; }

// gemm_f16_splitk: tight row-major fp16, the tile must divide the shape.
static int splitk_run(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C, void *ws,
                      size_t ws_bytes, int tile_id, int splits, int algo, cudaStream_t stream) {
    int rc = validate_common(M, N, K, A, B, C);
    if (rc) return rc;
    if (M == 0 || N == 0) return SDT_OK;
    if (!splitk_algo_ok(algo)) return fail(SDT_ERR_ARG, "unknown split-K algorithm %d", algo);
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    if (K == 0) return gemm_dispatch(M, N, K, A, B, C, reinterpret_cast<sdt_stream_t>(stream), -1, -1);
    if (tile_id < 0) {
        int sp = 1;
        rc = pick_splitk_for(M, N, K, dev.sm_count, dev.smem_optin, dev.smem_per_sm, &tile_id, &sp);
        if (rc) return rc;
        if (splits <= 0 && !is_streamk(algo)) splits = sp;
    }
    if (!splitk_tile_ok(tile_id)) return fail(SDT_ERR_TILE, "tile %d has no split-K form", tile_id);
    const LadderTile &t = kLadder[tile_id];
    if (!splitk_feasible(t, M, N, K, dev.smem_optin))
        return fail(SDT_ERR_TILE, "tile %s does not divide %lldx%lldx%lld", t.name, (long long)M, (long long)N,
                    (long long)K);
    if (is_streamk(algo))
        return streamk_launch_ex(tile_id, splits, algo, M, N, K, A, K, B, N, C, N, SDT_DTYPE_F16, 0, ws, ws_bytes,
                                 stream, dev);
    return splitk_launch_ex(tile_id, splits, algo, M, N, K, A, K, B, N, C, N, SDT_DTYPE_F16, 0, ws, ws_bytes, stream,
                            dev);
}

// (tile, splits) for split-K on any shape: the split-K cost model over the tiles
// with a split-K form that fit on chip (tiles may overhang ragged edges).
static int pick_splitk_any(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit, int smem_per_sm,
                           int *tile_out, int *splits_out) {
    double best = 0.0;
    int bt = -1, bs = 1;
    const int64_t nK = ceil_div(K, kBK);
    for (int i = 0; i < kNumTiles; ++i) {
        if (!splitk_tile_ok(i) || !kLadder[i].candidate || !fits_chip(kLadder[i], smem_limit)) continue;
        for (int sp = 1; sp <= 32 && sp <= nK; ++sp) {
            if (splitk_effective(nK, sp) != sp) continue;
            const double c = splitk_model_us(kLadder[i], M, N, K, sp, sm_count, smem_per_sm);
            if (bt < 0 || c < best * (1.0 - 1e-9)) {
                best = c;
                bt = i;
                bs = sp;
            }
        }
    }
    if (bt < 0) return fail(SDT_ERR_TILE, "no split-K tile fits this device");
    *tile_out = bt;
    *splits_out = bs;
    return SDT_OK;
}

// Argument checks of gemm_ex and gemm_ex_splitk (SDT_OK also for empty shapes).
static int validate_ex(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                       void *C, int64_t ldc, int dtype, int layout) {
    if (M < 0 || N < 0 || K < 0)
        return fail(SDT_ERR_SHAPE, "negative dimension (M=%lld N=%lld K=%lld)", (long long)M, (long long)N,
                    (long long)K);
    if (dtype != SDT_DTYPE_F16 && dtype != SDT_DTYPE_BF16) return fail(SDT_ERR_ARG, "unknown dtype %d", dtype);
    if (layout & ~(SDT_LAYOUT_A_T | SDT_LAYOUT_B_T)) return fail(SDT_ERR_ARG, "unknown layout flags %d", layout);
    if (M == 0 || N == 0) return SDT_OK;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return fail(SDT_ERR_SHAPE, "dimension above 2^30");
    if (!C || (K > 0 && (!A || !B))) return fail(SDT_ERR_NULL, "NULL operand pointer");
    if ((reinterpret_cast<uintptr_t>(C) & 15) ||
        (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))))
        return fail(SDT_ERR_ALIGN, "A, B and C must be 16-byte aligned");
    if (N % 8) return fail(SDT_ERR_SHAPE, "N must be a multiple of 8 (C rows are written 16 bytes at a time)");
    if (ldc < N || ldc % 8) return fail(SDT_ERR_ARG, "ldc must be >= N and a multiple of 8");
    if (K > 0) {
        const int64_t a_inner = (layout & SDT_LAYOUT_A_T) ? M : K;
        const int64_t b_inner = (layout & SDT_LAYOUT_B_T) ? K : N;
        if (lda < a_inner || lda % 8) return fail(SDT_ERR_ARG, "lda must be >= %lld and a multiple of 8", (long long)a_inner);
        if (ldb < b_inner || ldb % 8) return fail(SDT_ERR_ARG, "ldb must be >= %lld and a multiple of 8", (long long)b_inner);
    }
    return SDT_OK;
}

// C = 0 for K == 0 (the empty sum), row stride ldc.
static int zero_c(int64_t M, int64_t N, void *C, int64_t ldc, cudaStream_t stream, const DeviceInfo &dev) {
    const int64_t total = M * (N / 8);
    const unsigned blocks = unsigned(std::min<int64_t>((total + 255) / 256, int64_t(dev.sm_count) * 8));
    zero_fill_2d<<<blocks, 256, 0, stream>>>(static_cast<uint16_t *>(C), M, N, ldc);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SDT_OK : fail(SDT_ERR_LAUNCH, "zero fill failed: %s", cudaGetErrorString(e));
}

static int gemm_ex_impl(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                        void *C, int64_t ldc, int dtype, int layout, int tile_id, cudaStream_t stream,
                        const TailWs *tw = nullptr) {
    int rc = validate_ex(M, N, K, A, lda, B, ldb, C, ldc, dtype, layout);
    if (rc || M == 0 || N == 0) return rc;
    if (tile_id < -1 || tile_id >= kNumTiles) return fail(SDT_ERR_TILE, "unknown tile id %d", tile_id);
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    if (K == 0) return zero_c(M, N, C, ldc, stream, dev);
    if (tile_id < 0) tile_id = pick_any(M, N, K, dev.sm_count, dev.smem_optin, dev.smem_per_sm);
    if (tile_id < 0 || !fits_chip(kLadder[tile_id], dev.smem_optin))
        return fail(SDT_ERR_TILE, "no tile fits this device");
    return run_tile_ex(tile_id, -1, M, N, K, A, lda, B, ldb, C, ldc, dtype, layout, stream, dev, 0, 0, tw);
}

// The workspace every gemm_f16_ws / gemm_ex_ws call accepts on a GPU with sm_count SMs:
// the counter region and one 256 x 256 fp32 slot per SM pair (a last round has at most
// one item per pair).
static size_t gemm_ws_bytes(int sm_count) {
    return kCounterRegionBytes + size_t(std::max(sm_count / 2, 1)) * 256 * 256 * 4;
}

// Checks a gemm_*_ws workspace (nullptr: none) and fills `tw`.
static int tail_ws_arg(void *ws, size_t bytes, int req, const DeviceInfo &dev, TailWs *tw) {
    *tw = TailWs{nullptr, 0, 0};
    if (!ws) return SDT_OK;
    if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(SDT_ERR_ALIGN, "the workspace must be 256-byte aligned");
    if (bytes < gemm_ws_bytes(dev.sm_count))
        return fail(SDT_ERR_ARG, "workspace of %zu bytes; sdt_gemm_workspace_bytes() is %zu", bytes,
                    gemm_ws_bytes(dev.sm_count));
    if (req < -1 || req == 1 || req > kPairTailMaxSplits)
        return fail(SDT_ERR_ARG, "tail_splits must be -1, 0 or 2..%d", kPairTailMaxSplits);
    *tw = TailWs{ws, bytes, req};
    return SDT_OK;
}

static int gemm_ex_splitk_impl(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                               int64_t ldb, void *C, int64_t ldc, int dtype, int layout, void *ws, size_t ws_bytes,
                               int tile_id, int splits, int algo, cudaStream_t stream) {
    int rc = validate_ex(M, N, K, A, lda, B, ldb, C, ldc, dtype, layout);
    if (rc || M == 0 || N == 0) return rc;
    if (!splitk_algo_ok(algo)) return fail(SDT_ERR_ARG, "unknown split-K algorithm %d", algo);
    if (tile_id < -1 || tile_id >= kNumTiles) return fail(SDT_ERR_TILE, "unknown tile id %d", tile_id);
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc) return rc;
    if (K == 0) return zero_c(M, N, C, ldc, stream, dev);
    if (tile_id < 0) {
        int sp = 1;
        rc = pick_splitk_any(M, N, K, dev.sm_count, dev.smem_optin, dev.smem_per_sm, &tile_id, &sp);
        if (rc) return rc;
        if (splits <= 0 && !is_streamk(algo)) splits = sp;
    }
    if (!splitk_tile_ok(tile_id)) return fail(SDT_ERR_TILE, "tile %d has no split-K form", tile_id);
    if (!fits_chip(kLadder[tile_id], dev.smem_optin)) return fail(SDT_ERR_TILE, "tile %d does not fit", tile_id);
    if (is_streamk(algo))
        return streamk_launch_ex(tile_id, splits, algo, M, N, K, A, lda, B, ldb, C, ldc, dtype, layout, ws, ws_bytes,
                                 stream, dev);
    return splitk_launch_ex(tile_id, splits, algo, M, N, K, A, lda, B, ldb, C, ldc, dtype, layout, ws, ws_bytes,
                            stream, dev);
}

// Entry for other translation units of the library (the no-allocation variant):
// the same validation and launches as gemm_f16_splitk on a given workspace.
int splitk_launch(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C, void *ws,
                  size_t ws_bytes, int tile_id, int splits, int algo, cudaStream_t stream) {
    return splitk_run(M, N, K, A, B, C, ws, ws_bytes, tile_id, splits, algo, stream);
}

}  // namespace sdt

using namespace sdt;

extern "C" {

int gemm_f16(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C, sdt_stream_t stream) {
    return gemm_dispatch(M, N, K, A, B, C, stream, -1, -1);
}

int gemm_f16_with_tile(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                       sdt_stream_t stream, int tile_id, int stagger) {
    if (tile_id < 0 || tile_id >= kNumTiles) {
        clear_error();
        return fail(SDT_ERR_TILE, "unknown tile id %d", tile_id);
    }
    return gemm_dispatch(M, N, K, A, B, C, stream, tile_id, stagger);
}

int gemm_f16_ws(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C, void *workspace,
                size_t workspace_bytes, sdt_stream_t stream) {
    clear_error();
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    TailWs tw;
    rc = tail_ws_arg(workspace, workspace_bytes, -1, dev, &tw);
    if (rc) return rc;
    return gemm_dispatch(M, N, K, A, B, C, stream, -1, -1, &tw);
}

int gemm_ex_ws(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
               int64_t ldc, int dtype, int layout, int tile_id, int tail_splits, void *workspace,
               size_t workspace_bytes, sdt_stream_t stream) {
    clear_error();
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    TailWs tw;
    rc = tail_ws_arg(workspace, workspace_bytes, tail_splits, dev, &tw);
    if (rc) return rc;
    return gemm_ex_impl(M, N, K, A, lda, B, ldb, C, ldc, dtype, layout, tile_id,
                        reinterpret_cast<cudaStream_t>(stream), &tw);
}

size_t sdt_gemm_workspace_bytes_for(int sm_count) {
    clear_error();
    return sm_count > 0 ? gemm_ws_bytes(sm_count) : 0;
}

size_t sdt_gemm_workspace_bytes(void) {
    DeviceInfo dev;
    if (current_device(&dev)) return 0;
    clear_error();
    return gemm_ws_bytes(dev.sm_count);
}

int sdt_pair_tail_plan(int64_t M, int64_t N, int64_t K, int tile_id, int sm_count, int smem_limit,
                       int with_workspace, int tail_splits, int *tail_start, int *num_items, int *splits,
                       int *split0_ktiles) {
    clear_error();
    if (!tail_start || !num_items || !splits || !split0_ktiles)
        return fail(SDT_ERR_NULL, "output pointers must not be NULL");
    if (tile_id < 0 || tile_id >= kNumTiles || kLadder[tile_id].cta_group != 2)
        return fail(SDT_ERR_TILE, "tile %d is not a two-CTA tile", tile_id);
    if (!dims_in_range(M, N, K) || sm_count < 2 || smem_limit <= 0)
        return fail(SDT_ERR_ARG, "dimensions and sm_count out of range");
    if (tail_splits < -1 || tail_splits == 1 || tail_splits > kPairTailMaxSplits)
        return fail(SDT_ERR_ARG, "tail_splits must be -1, 0 or 2..%d", kPairTailMaxSplits);
    const LadderTile &t = kLadder[tile_id];
    const int64_t tiles = ceil_div(M, t.BM) * ceil_div(N, t.BN);
    if (tiles > kMaxGridTiles) return fail(SDT_ERR_SHAPE, "grid too large");
    const PairTail pt = pair_tail_plan(t, int(tiles), int(ceil_div(K, kBK)), sm_count / 2,
                                       tile_stages(t, smem_limit), with_workspace != 0, tail_splits);
    *tail_start = pt.tail_start;
    *num_items = pt.num_items;
    *splits = pt.splits;
    *split0_ktiles = pt.long_k;
    return SDT_OK;
}

int sdt_num_tiles(void) { return kNumTiles; }

int sdt_tile_info(int tile_id, sdt_tile_desc *out) {
    clear_error();
    if (!out) return fail(SDT_ERR_NULL, "out is NULL");
    if (tile_id < 0 || tile_id >= kNumTiles) return fail(SDT_ERR_TILE, "unknown tile id %d", tile_id);
    const LadderTile &t = kLadder[tile_id];
    memset(out, 0, sizeof *out);
    out->id = tile_id;
    out->BM = t.BM;
    out->BN = t.BN;
    out->BK = kBK;
    out->cta_group = t.cta_group;
    out->stages = t.stages;
    out->threads = t.threads;
    out->smem_bytes = tile_smem(t, t.stages);
    out->tmem_cols = t.tmem_cols;
    snprintf(out->name, sizeof out->name, "%s", t.name);
    return SDT_OK;
}

const char *sdt_tile_name(int tile_id) {
    if (tile_id < 0 || tile_id >= kNumTiles) return nullptr;
    return kLadder[tile_id].name;
}

int sdt_feasible_tiles_for(int64_t M, int64_t N, int64_t K, int smem_limit, int *ids, int cap) {
    clear_error();
    if (cap < 0 || (cap > 0 && !ids)) return fail(SDT_ERR_NULL, "ids is NULL with cap > 0");
    int n = 0;
    for (int i = 0; i < kNumTiles; ++i) {
        if (!feasible(kLadder[i], M, N, K, smem_limit)) continue;
        if (n < cap) ids[n] = i;
        ++n;
    }
    return n;
}

int sdt_feasible_tiles(int64_t M, int64_t N, int64_t K, int *ids, int cap) {
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return sdt_feasible_tiles_for(M, N, K, dev.smem_optin, ids, cap);
}

double sdt_tile_estimate_us(int tile_id, int64_t M, int64_t N, int64_t K, int sm_count) {
    clear_error();
    if (tile_id < 0 || tile_id >= kNumTiles) return fail(SDT_ERR_TILE, "unknown tile id %d", tile_id);
    if (sm_count <= 0 || M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return fail(SDT_ERR_ARG, "dimensions must be in 1..2^30 and sm_count positive");
    return model_us(kLadder[tile_id], M, N, K, sm_count, 233472);
}

int sdt_pick_tile_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit) {
    clear_error();
    if (sm_count <= 0) return fail(SDT_ERR_ARG, "sm_count must be positive");
    // Shared memory per SM on sm_100-class parts is 228 KiB.
    const int id = pick_for(M, N, K, sm_count, smem_limit, 233472);
    if (id < 0) return fail(SDT_ERR_SHAPE, "no feasible tile");
    return id;
}

int sdt_pick_tile(int64_t M, int64_t N, int64_t K) {
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    clear_error();
    const int id = pick_for(M, N, K, dev.sm_count, dev.smem_optin, dev.smem_per_sm);
    if (id < 0) return fail(SDT_ERR_SHAPE, "no feasible tile");
    return id;
}

int sdt_seed_tile(int64_t M, int64_t N, int units) {
    clear_error();
    if (units <= 0 || M < 0 || N < 0) return fail(SDT_ERR_ARG, "bad arguments");
    const int64_t blocks = (M / 128) * (N / 128);
    const char *name = blocks >= units ? "128x128" : (3 * blocks >= 2 * int64_t(units) ? "64x128" : "64x64");
    return find_tile(name);
}

int sdt_load_tune_table(const char *path) {
    clear_error();
    if (!path) return fail(SDT_ERR_NULL, "path is NULL");
    std::map<ShapeKey, TuneEntry> tab;
    int rc = load_table_file(path, &tab);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_table_mu);
    g_table = std::move(tab);
    return SDT_OK;
}

void sdt_clear_tune_table(void) {
    std::lock_guard<std::mutex> lock(g_table_mu);
    g_table.clear();
}

int sdt_tune_table_size(void) {
    std::lock_guard<std::mutex> lock(g_table_mu);
    return int(g_table.size());
}

int sdt_tune_table_lookup(int64_t M, int64_t N, int64_t K) {
    TuneEntry e;
    return table_lookup(M, N, K, &e) ? e.tile : -1;
}

int gemm_ex(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
            int64_t ldc, int dtype, int layout, int tile_id, sdt_stream_t stream) {
    clear_error();
    return gemm_ex_impl(M, N, K, A, lda, B, ldb, C, ldc, dtype, layout, tile_id, reinterpret_cast<cudaStream_t>(stream));
}

int sdt_pick_tile_any_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit) {
    clear_error();
    if (sm_count <= 0 || M <= 0 || N <= 0 || K <= 0) return fail(SDT_ERR_ARG, "dimensions and sm_count must be positive");
    const int id = pick_any(M, N, K, sm_count, smem_limit, 233472);
    return id >= 0 ? id : fail(SDT_ERR_SHAPE, "no tile fits");
}

size_t sdt_splitk_workspace_bytes(int64_t M, int64_t N, int64_t K, int tile_id, int splits) {
    clear_error();
    if (M <= 0 || N <= 0 || K <= 0 || !splitk_tile_ok(tile_id) || splits < 1) return 0;
    const LadderTile &t = kLadder[tile_id];
    if (t.swap || M % t.BM || N % t.BN || K % kBK || splits > K / kBK) return 0;
    return splitk_ws_bytes(t, M, N, K, splits);
}

int sdt_splitk_workspace_init(void *workspace, size_t workspace_bytes, sdt_stream_t stream) {
    clear_error();
    if (!workspace) return fail(SDT_ERR_NULL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(SDT_ERR_ALIGN, "the workspace must be 256-byte aligned");
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    const size_t n = workspace_bytes / 4;
    if (n == 0) return SDT_OK;
    const unsigned blocks = unsigned(std::min<size_t>((n + 255) / 256, size_t(dev.sm_count) * 8));
    zero_fill_u32<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<unsigned *>(workspace), n);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SDT_OK : fail(SDT_ERR_LAUNCH, "workspace init failed: %s", cudaGetErrorString(e));
}

int sdt_pick_splitk_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit, int *tile_id, int *splits) {
    clear_error();
    if (!tile_id || !splits) return fail(SDT_ERR_NULL, "tile_id and splits must not be NULL");
    if (sm_count <= 0) return fail(SDT_ERR_ARG, "sm_count must be positive");
    return pick_splitk_for(M, N, K, sm_count, smem_limit, 233472, tile_id, splits);
}

int gemm_ex_splitk(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                   int64_t ldc, int dtype, int layout, void *workspace, size_t workspace_bytes, int tile_id, int splits,
                   int algo, sdt_stream_t stream) {
    clear_error();
    return gemm_ex_splitk_impl(M, N, K, A, lda, B, ldb, C, ldc, dtype, layout, workspace, workspace_bytes, tile_id,
                               splits, algo, reinterpret_cast<cudaStream_t>(stream));
}

size_t sdt_splitk_ex_workspace_bytes(int64_t M, int64_t N, int64_t K, int tile_id, int splits) {
    clear_error();
    if (!splitk_tile_ok(tile_id)) return 0;
    const LadderTile &t = kLadder[tile_id];
    return t.swap ? splitk_ws_bytes(t, N, M, K, splits) : splitk_ws_bytes(t, M, N, K, splits);
}

size_t sdt_streamk_workspace_bytes(int64_t M, int64_t N, int64_t K, int tile_id, int ctas) {
    clear_error();
    if (!streamk_tile_ok(tile_id)) return 0;
    const LadderTile &t = kLadder[tile_id];
    return t.swap ? streamk_ws_bytes(t, N, M, K, ctas) : streamk_ws_bytes(t, M, N, K, ctas);
}
int sdt_streamk_ctas_for(int tile_id, int sm_count, int smem_limit) {
    clear_error();
    if (!streamk_tile_ok(tile_id)) return fail(SDT_ERR_TILE, "tile %d has no stream-K form", tile_id);
    if (sm_count <= 0 || smem_limit <= 0) return fail(SDT_ERR_ARG, "sm_count and smem_limit must be positive");
    return sm_count * streamk_ctas_per_sm(kLadder[tile_id], smem_limit, 233472);
}
int sdt_streamk_ctas(int tile_id) {
    clear_error();
    if (!streamk_tile_ok(tile_id)) return fail(SDT_ERR_TILE, "tile %d has no stream-K form", tile_id);
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return dev.sm_count * streamk_ctas_per_sm(kLadder[tile_id], dev.smem_optin, dev.smem_per_sm);
}
int sdt_pick_splitk_any_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit, int *tile_id,
                            int *splits) {
    clear_error();
    if (!tile_id || !splits) return fail(SDT_ERR_NULL, "tile_id and splits must not be NULL");
    if (sm_count <= 0 || M <= 0 || N <= 0 || K <= 0) return fail(SDT_ERR_ARG, "dimensions and sm_count must be positive");
    return pick_splitk_any(M, N, K, sm_count, smem_limit, 233472, tile_id, splits);
}

int gemm_f16_splitk(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C, void *workspace,
                    size_t workspace_bytes, int tile_id, int splits, int algo, sdt_stream_t stream) {
    clear_error();
    return splitk_run(M, N, K, A, B, C, workspace, workspace_bytes, tile_id, splits, algo,
                      reinterpret_cast<cudaStream_t>(stream));
}

// Number of tensor maps encoded so far (cache misses); for the cache-key tests.
int64_t sdt_debug_tensor_map_encodes(void) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    return int64_t(g_map_encodes);
}

}  // extern "C"
