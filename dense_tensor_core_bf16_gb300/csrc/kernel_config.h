// Compile-time shapes of the GEMM kernel variants, shared by the planner (host
// C++) and the CUDA sources.
//
// A variant is (CTA group, BN):
//   * CTA group 1: one CTA computes a 128 x BN block of C with
//     tcgen05.mma.cta_group::1 (M = 128);
//   * CTA group 2: a cluster of two CTAs on a pair of SMs computes a
//     256 x BN block with tcgen05.mma.cta_group::2 (M = 256): each CTA stages
//     its own 128 rows of A and BN/2 rows of B, and holds its 128 rows of the
//     accumulator in its own tensor memory.
// Operands arrive in k-tiles of 64 or 128 bf16 (one or two 128-byte swizzle
// spans, loaded as one TMA box each) through a ring of as many stages as the
// shared memory holds.  One k-tile is one wait on the ring and one commit by
// the MMA thread: 128-wide k-tiles give the Tensor Core 8 MMAs per wait, which
// it needs to stay busy (4 per wait leaves it idle about a tenth of the time).
#pragma once

#if defined(__CUDACC__)
#define GEMM_HD __host__ __device__
#else
#define GEMM_HD
#endif

namespace gemm {

constexpr int TILE_K = 64;                // bf16 per TMA box row: 128 bytes, one swizzle span
constexpr int MMA_K = 16;                 // K of one kind::f16 tcgen05.mma
constexpr int CTA_ROWS = 128;             // rows of C per CTA = TMEM lanes
constexpr int ACC_BUFS = 2;               // accumulators in TMEM (epilogue overlaps the next tile)
constexpr int NUM_WARPS = 6;              // 0: TMA producer, 1: TMEM owner + MMA issuer, 2..5: epilogue
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int EPI_WARPS = 4;
// accumulator full/empty, drain, and per epilogue warp two loads of previous
// C into its staging buffers (the fused epilogue with beta != 0); + 2 per stage
constexpr int NUM_BARRIERS_FIXED = 2 * ACC_BUFS + 1 + 2 * 4;
constexpr int SMEM_LIMIT = 232448;        // opt-in dynamic shared memory per CTA on sm_100-class parts
constexpr int MAX_STAGES = 8;
// Epilogue staging: per epilogue warp, two buffers of one 32 x 32 chunk of C
// (fp32 at most: 4 KiB), which TMA stores to global memory.
constexpr int EPI_BUF_BYTES = 4096;
constexpr int EPI_STAGING_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;

enum Variant : int {
    VARIANT_AUTO = 0,
    VARIANT_1SM_128x256 = 1,
    VARIANT_2SM_256x256 = 2,
    VARIANT_2SM_256x128 = 3,
    VARIANT_1SM_128x128 = 4,
    VARIANT_COUNT = 5
};

GEMM_HD constexpr int pow2_at_least(int x, int p = 32) { return p >= x ? p : pow2_at_least(x, p * 2); }

struct VariantInfo {
    int cta_group;   // CTAs cooperating on one tile (cluster size)
    int bn;          // columns of C per tile
    int tile_k;      // K per k-tile (a multiple of TILE_K)
    int k_boxes;     // TMA boxes per operand per k-tile (tile_k / TILE_K)
    int tile_m;      // rows of C per tile (128 * cta_group)
    int b_rows;      // rows of B (N direction) each CTA stages
    int a_stage;     // bytes of A per stage per CTA
    int b_stage;     // bytes of B per stage per CTA
    int stage;       // a_stage + b_stage
    int stages;      // ring depth
    int smem;        // dynamic shared memory per CTA
    int tmem_cols;   // tensor-memory columns per CTA (power of two >= 32)
};

GEMM_HD constexpr VariantInfo make_variant(int cg, int bn, int tk) {
    const int a = CTA_ROWS * tk * 2;
    const int b = (bn / cg) * tk * 2;
    const int st = a + b;
    const int fixed = 1024 + (NUM_BARRIERS_FIXED + 2 * MAX_STAGES) * 8 + 16;
    int stages = (SMEM_LIMIT - fixed - EPI_STAGING_BYTES) / st;
    if (stages > MAX_STAGES) stages = MAX_STAGES;
    return VariantInfo{cg, bn, tk, tk / TILE_K, CTA_ROWS * cg, bn / cg, a, b, st, stages,
                       1024 + stages * st + EPI_STAGING_BYTES + (NUM_BARRIERS_FIXED + 2 * stages) * 8 + 16,
                       pow2_at_least(ACC_BUFS * bn)};
}

GEMM_HD constexpr VariantInfo variant_info(int v) {
    return v == VARIANT_2SM_256x256 ? make_variant(2, 256, 128)
         : v == VARIANT_2SM_256x128 ? make_variant(2, 128, 64)
         : v == VARIANT_1SM_128x128 ? make_variant(1, 128, 64)
                                    : make_variant(1, 256, 64);
}

static_assert(variant_info(VARIANT_1SM_128x256).stages == 4, "1-SM 128x256: four 48 KiB stages");
static_assert(variant_info(VARIANT_2SM_256x256).stages == 3, "2-SM 256x256: three 64 KiB stages");
static_assert(variant_info(VARIANT_2SM_256x256).smem <= SMEM_LIMIT, "fits");
static_assert(variant_info(VARIANT_2SM_256x128).smem <= SMEM_LIMIT, "fits");

constexpr int DEFAULT_RASTER_GROUP_M = 16;
constexpr int MANY_WAVES = 8;                  // tiles >= this many waves of clusters ...
constexpr int MANY_WAVES_RASTER_GROUP_M = 8;   // ... take raster groups of 8 m-tiles
constexpr int DEFAULT_TIMEOUT_MS = 4000;
// The default limit also grows with the longest stretch of main loop a single
// wait can span (the epilogue's wait for a whole unit's accumulator, a
// stream-K owner's wait for its contributors): this much per k-tile, about
// 16 times what a 128-wide k-tile of the pair kernel takes at full clock.
constexpr int DEFAULT_TIMEOUT_US_PER_K_TILE = 8;
constexpr int MIN_K_TILES_PER_SPLIT = 4;  // automatic split-K keeps at least this many k-tiles per slice
// Handing partial tiles between CTAs (split-K's fp32 slices and combine
// kernel, stream-K's fix-ups) costs a roughly fixed 5-25 us on GB300, which
// only a long enough K repays (measured over tile counts 2-256 and K 1k-16k).
// The plan's own choice therefore splits K only for few tiles: tiles * 8 <=
// resident clusters with K >= AUTO_SPLIT_MIN_K, or tiles * 4 <= clusters with
// K >= LONG_K; and spreads a tail of tiles over the clusters (stream-K) only
// with at least one full wave, when the partly filled last wave would leave
// at least STREAM_K_MIN_WASTE 128-wide k-tiles of a 128 x 256 block per SM
// idle in the average cluster.
constexpr long long AUTO_SPLIT_MIN_K = 2048;
constexpr long long LONG_K = 6144;
constexpr double STREAM_K_MIN_WASTE = 12.0;
// The stream-K tail's range boundaries travel in the kernel's parameters, one
// per cluster; a launch with more clusters than this takes no tail.
constexpr int SK_MAX_CLUSTERS = 160;

}  // namespace gemm
