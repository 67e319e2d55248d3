// gemm_bf16.cu -- BF16 Tensor Core GEMM for GB300 (sm_103a): kernels and the
// C-ABI launcher.  Contract: include/gemm_bf16.h.
//
// Method (chapter 10 "Tensor Cores, shapes, and tile alignment"; lesson
// "The Tensor Core"; post "Grid 24 is not headroom"):
//   * two-sided tiling: A and B tiles are staged once in shared memory and
//     reused by every MMA of the tile -- keeping the Tensor Cores supplied
//     with operands is what limits them;
//   * the staging is a ring of STAGES slots filled by TMA and guarded by
//     mbarriers -- at one CTA per SM, pipeline depth is the only way to hide
//     memory latency, and it is bought with shared memory;
//   * warp specialisation: one producer warp issues the TMA copies, one warp
//     issues tcgen05.mma into an fp32 accumulator in tensor memory (TMEM),
//     four warps drain finished accumulators to global memory;
//   * a persistent grid of min(G, S b) CTAs loops over the work units; two
//     TMEM accumulators let the epilogue of one tile overlap the main loop of
//     the next;
//   * split-K: a work unit is a (tile, K-slice) pair; slices write fp32
//     partial sums to a separate buffer that a combine kernel adds in slice
//     order;
//   * ragged M, N, K: TMA zero-fills out-of-range operand elements and the
//     epilogue masks out-of-range stores.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_bf16.h"
#include "kernel_config.h"
#include "plan_internal.h"
#include "ptx.cuh"

namespace gemm {

// Bit set of the pipeline waits that ran out of time (see gemm_get_device_status).
__device__ unsigned int g_fault_word;

enum : unsigned {
    SITE_PRODUCER = 1u,
    SITE_MMA_OPERANDS = 2u,
    SITE_MMA_ACC = 4u,
    SITE_EPI_ACC = 8u,
    SITE_DRAIN = 16u,
    SITE_FIXUP = 32u,
    SITE_EPI_C = 64u
};

struct KernelParams {
    int M, N, K;
    int tiles_m, tiles_n;
    int k_tiles;                 // ceil(K / k-tile width of the variant)
    int split_k;
    int group_m;                 // m-tiles per raster group
    long long num_units;         // tiles * split_k
    void *out;                   // C
    long long ld_out;            // leading dimension of C, elements
    int out_bf16;                // 1: bf16 stores, 0: fp32 stores
    int n_tma;                   // columns of C stored by TMA: N rounded down to whole 16-byte pieces
    unsigned long long timeout_ns;
    int skip_load;               // test hook (0 = off)
    int a_mn, b_mn;              // 1: the operand is MN-major in memory (A column-major, B row-major)
    // Implicit-GEMM convolution (conv = 1): row m of A is output pixel
    // m = (n, p, q) of an N x P x Q output; box i (64 wide) of the GEMM's K is
    // filter tap i / ncb (r = tap / S, s = tap % S), channels 64 (i % ncb) on.
    // tmap_a is an im2col map of x (NHWC): a box is the 128 pixels of the
    // CTA's rows at one tap; tmap_b is the filter (KRSC) as a 3-D map
    // (channels, taps, output channels).
    int conv;
    int cv_S, cv_PQ, cv_Q, cv_taps;
    int pad_h, pad_w, str_h, str_w, dil_h, dil_w;
    int ncb;
    // fused epilogue (epi = 1): C := act(alpha * acc + beta * C + bias[n])
    int epi;
    float alpha, beta;
    const float *bias;           // N values or nullptr
    int act;                     // gemm_activation_t
    // Stream-K tail (sk_tiles > 0; split_k is then 1): tiles [0, dp_tiles) are
    // computed whole, round robin over the clusters; the k-iterations of tiles
    // [dp_tiles, tiles) are dealt out to the clusters in the contiguous ranges
    // of sk_bounds, which the clusters run first.
    int num_clusters;            // clusters launched (gridDim.x / CTA group)
    int dp_tiles;
    int sk_tiles;
    long long sk_iters;          // sk_tiles * k_tiles (the last of sk_bounds)
    // fp32 partial tiles, one slot of tile rows x BN each: with split-K,
    // [split][tile] (slot split * tiles + tile); with a stream-K tail, one
    // slot per cluster.  Slots are laid out warp-major (see the epilogue).
    float *partials;
    unsigned int *sk_flags;      // [num_clusters][CTA group][4 epilogue warps]
    unsigned int epoch;          // value the flags of this launch carry (never 0)
    // first stream-K iteration of cluster c (c = 0 .. num_clusters; the last
    // is sk_iters), as the plan deals them out
    long long sk_bounds[SK_MAX_CLUSTERS + 1];
};

// Wait for the phase of `bar` with parity `parity`.  Gives up after
// `timeout_ns` (recording `site` in the fault word and raising the CTA's abort
// flag), or -- when `honor_abort` -- as soon as another role has given up.
// CLUSTER_SCOPE: acquire at cluster scope (barriers the peer CTA signals).
template <bool CLUSTER_SCOPE>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           unsigned long long timeout_ns, unsigned site, bool honor_abort) {
    auto try_wait = [&]() {
        return CLUSTER_SCOPE ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (try_wait()) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (try_wait()) return true;
        if ((i & 31u) == 0) {
            if (honor_abort && *abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                atomicOr(&g_fault_word, site);
                return false;
            }
        }
    }
}

enum : int { KIND_FULL = 0, KIND_PARTIAL = 1, KIND_OWNER = 2 };

struct Unit {
    int tm, tn;         // tile coordinates (in tiles)
    int split;          // K slice
    int kb_begin;       // first k-tile of the slice
    int kb_count;       // k-tiles in the slice (>= 1)
    int kind;           // KIND_FULL: store C (or the split-K slice); stream-K only:
                        // KIND_PARTIAL: a segment not starting at k = 0, stored to this
                        // cluster's partial slot; KIND_OWNER: the k = 0 segment of a tile
                        // whose later segments other clusters computed
    int sk_tile;        // index of the tile in the stream-K region (stream-K units)
};

// Work unit u -> tile and K slice.  Tiles are visited in groups of group_m
// tile-rows, column by column inside a group, so that the tiles in flight at
// one time share A rows and B columns in L2.  Slices split the k-tiles as
// evenly as possible: the first (k_tiles mod split_k) slices get one more.
__device__ __forceinline__ Unit decode_unit(long long u, const KernelParams &p) {
    Unit w;
    const long long tile = u / p.split_k;
    w.split = static_cast<int>(u - tile * p.split_k);
    const long long per_group = static_cast<long long>(p.group_m) * p.tiles_n;
    const int group = static_cast<int>(tile / per_group);
    const int first_m = group * p.group_m;
    const int gsize = min(p.tiles_m - first_m, p.group_m);
    const int r = static_cast<int>(tile - static_cast<long long>(group) * per_group);
    w.tm = first_m + r % gsize;
    w.tn = r / gsize;
    const int base = p.k_tiles / p.split_k;
    const int rem = p.k_tiles - base * p.split_k;
    w.kb_count = base + (w.split < rem ? 1 : 0);
    w.kb_begin = w.split * base + min(w.split, rem);
    w.kind = KIND_FULL;
    w.sk_tile = -1;
    return w;
}

// Tile index -> tile coordinates, grouped raster (see decode_unit).
__device__ __forceinline__ void tile_coords(long long tile, const KernelParams &p, int &tm, int &tn) {
    const long long per_group = static_cast<long long>(p.group_m) * p.tiles_n;
    const int group = static_cast<int>(tile / per_group);
    const int first_m = group * p.group_m;
    const int gsize = min(p.tiles_m - first_m, p.group_m);
    const int r = static_cast<int>(tile - static_cast<long long>(group) * per_group);
    tm = first_m + r % gsize;
    tn = r / gsize;
}

// First stream-K iteration of cluster c (c = num_clusters: the end).
__device__ __forceinline__ long long sk_range_start(const KernelParams &p, long long c) { return p.sk_bounds[c]; }

// The work of one cluster, in the order every role of its CTAs walks it:
// its stream-K range (cut at tile boundaries), then its whole tiles.
struct Schedule {
    long long it, it_end;   // stream-K iterations still to do
    long long u;            // next whole-tile (or split-K) unit
    long long cluster;

    __device__ __forceinline__ Schedule(const KernelParams &p, long long c) : u(c), cluster(c) {
        if (p.sk_tiles > 0) {
            it = sk_range_start(p, c);
            it_end = sk_range_start(p, c + 1);
        } else {
            it = it_end = 0;
        }
    }

    __device__ __forceinline__ bool next(const KernelParams &p, Unit &w) {
        if (it < it_end) {
            const long long t = it / p.k_tiles;
            const int k0 = static_cast<int>(it - t * p.k_tiles);
            const long long left = it_end - it;
            const int k1 = static_cast<int>(min(static_cast<long long>(p.k_tiles), k0 + left));
            tile_coords(p.dp_tiles + t, p, w.tm, w.tn);
            w.split = 0;
            w.kb_begin = k0;
            w.kb_count = k1 - k0;
            w.kind = k0 > 0 ? KIND_PARTIAL : (k1 < p.k_tiles ? KIND_OWNER : KIND_FULL);
            w.sk_tile = static_cast<int>(t);
            it += k1 - k0;
            return true;
        }
        const long long units = p.sk_tiles > 0 ? p.dp_tiles : p.num_units;
        if (u < units) {
            w = decode_unit(u, p);
            u += p.num_clusters;
            return true;
        }
        return false;
    }
};

// ---- the fused epilogue ----------------------------------------------------
//
// act(alpha * acc + beta * c + b) in fp32, each operation rounded as written
// (no contraction): the tolerance the tests hold it to counts those roundings.
//
// GELU is v * Phi(v) with Phi(v) = erfc(-v / sqrt 2) / 2.  erfc comes from
// the rational approximation of Abramowitz & Stegun, Handbook of Mathematical
// Functions, formula 7.1.26 (after Hastings): for z >= 0,
//     erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2) + e(z),
//     t = 1 / (1 + p z),  |e(z)| <= 1.5e-7.
// With z = |v| / sqrt 2 and E = erfc(z) / 2 (the a_k halved, which is exact):
//     v >= 0:  v Phi(v) = v - v E = v (1 - E)      v < 0:  v Phi(v) = v E,
// and as 0 < E <= 1/2, both cases are max(v E, v (1 - E)): no branch, no
// select on the sign.  1 + p z is fma(|v|, p / sqrt 2, 1), and exp(-z^2) is
// 2^(v^2 * (-log2(e) / 2)).  With the reciprocal and the power of two each
// within a few ulps, Phi is within about 5e-7, so v Phi(v) is within 2^-20 |v| --
// inside the stated tolerance.  gelu2 evaluates two values with the paired
// instructions; gelu is the same operations on one value, so both give the
// same bits.
namespace gelu_as {
constexpr float P_SQRT1_2 = static_cast<float>(0.3275911 / 1.4142135623730951);   // p / sqrt 2
constexpr float HALF_A1 = 0.5f * 0.254829592f, HALF_A2 = 0.5f * -0.284496736f, HALF_A3 = 0.5f * 1.421413741f,
                HALF_A4 = 0.5f * -1.453152027f, HALF_A5 = 0.5f * 1.061405429f;
constexpr float NEG_HALF_LOG2E = static_cast<float>(-0.5 * 1.4426950408889634);
}  // namespace gelu_as

__device__ __forceinline__ float gelu(float v) {
    using namespace gelu_as;
    const float t = ptx::rcp_approx(fmaf(fabsf(v), P_SQRT1_2, 1.0f));
    float q = fmaf(t, HALF_A5, HALF_A4);
    q = fmaf(t, q, HALF_A3);
    q = fmaf(t, q, HALF_A2);
    q = fmaf(t, q, HALF_A1);
    q = __fmul_rn(q, t);
    const float e = __fmul_rn(q, ptx::ex2_approx(__fmul_rn(__fmul_rn(v, v), NEG_HALF_LOG2E)));   // E
    const float one_minus_e = fmaf(e, -1.0f, 1.0f);
    return fmaxf(__fmul_rn(v, e), __fmul_rn(v, one_minus_e));
}

// gelu of both halves of a pair
__device__ __forceinline__ uint64_t gelu2(uint64_t v) {
    using namespace gelu_as;
    uint32_t v0, v1;
    ptx::f2_unpack(v, v0, v1);
    const uint64_t d = ptx::f2_fma(ptx::f2_pack(v0 & 0x7FFFFFFFu, v1 & 0x7FFFFFFFu), ptx::f2_splat(P_SQRT1_2),
                                   ptx::f2_splat(1.0f));
    uint32_t d0, d1;
    ptx::f2_unpack(d, d0, d1);
    const uint64_t t = ptx::f2_pack(__float_as_uint(ptx::rcp_approx(__uint_as_float(d0))),
                                    __float_as_uint(ptx::rcp_approx(__uint_as_float(d1))));
    uint64_t q = ptx::f2_fma(t, ptx::f2_splat(HALF_A5), ptx::f2_splat(HALF_A4));
    q = ptx::f2_fma(t, q, ptx::f2_splat(HALF_A3));
    q = ptx::f2_fma(t, q, ptx::f2_splat(HALF_A2));
    q = ptx::f2_fma(t, q, ptx::f2_splat(HALF_A1));
    q = ptx::f2_mul(q, t);
    const uint64_t w = ptx::f2_mul(ptx::f2_mul(v, v), ptx::f2_splat(NEG_HALF_LOG2E));
    uint32_t w0, w1;
    ptx::f2_unpack(w, w0, w1);
    const uint64_t e = ptx::f2_mul(q, ptx::f2_pack(__float_as_uint(ptx::ex2_approx(__uint_as_float(w0))),
                                                   __float_as_uint(ptx::ex2_approx(__uint_as_float(w1)))));
    const uint64_t one_minus_e = ptx::f2_fma(e, ptx::f2_splat(-1.0f), ptx::f2_splat(1.0f));
    uint32_t h0, h1, y0, y1;
    ptx::f2_unpack(ptx::f2_mul(v, e), h0, h1);
    ptx::f2_unpack(ptx::f2_mul(v, one_minus_e), y0, y1);
    return ptx::f2_pack(__float_as_uint(fmaxf(__uint_as_float(h0), __uint_as_float(y0))),
                        __float_as_uint(fmaxf(__uint_as_float(h1), __uint_as_float(y1))));
}

// alpha * acc + beta * c + b, then ReLU when asked (GELU is applied apart).
__device__ __forceinline__ float epilogue_linear(float acc, float c, float b, float alpha, float beta, int act) {
    float v = __fmul_rn(alpha, acc);
    v = __fadd_rn(v, __fmul_rn(beta, c));
    v = __fadd_rn(v, b);
    return act == GEMM_ACT_RELU ? fmaxf(v, 0.0f) : v;
}

__device__ __forceinline__ float epilogue_value(float acc, float c, float b, float alpha, float beta, int act) {
    const float v = epilogue_linear(acc, c, b, alpha, beta, act);
    return act == GEMM_ACT_GELU ? gelu(v) : v;
}

// Four consecutive previous values of C at (row, col) .. (row, col+3), as
// fp32; entries at n >= N read as 0 (they are never stored).
__device__ __forceinline__ float4 load_c4(const void *C, long long ldc, int out_bf16, int row, int col, int N) {
    float e[4] = {0.f, 0.f, 0.f, 0.f};
    if (out_bf16) {
        const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(C) + static_cast<long long>(row) * ldc + col;
        if (col + 4 <= N) {
            const uint2 u = *reinterpret_cast<const uint2 *>(src);
            e[0] = __uint_as_float(u.x << 16);
            e[1] = __uint_as_float(u.x & 0xFFFF0000u);
            e[2] = __uint_as_float(u.y << 16);
            e[3] = __uint_as_float(u.y & 0xFFFF0000u);
        } else {
            for (int j = 0; j < 4 && col + j < N; ++j) e[j] = __bfloat162float(src[j]);
        }
    } else {
        const float *src = static_cast<const float *>(C) + static_cast<long long>(row) * ldc + col;
        if (col + 4 <= N) return *reinterpret_cast<const float4 *>(src);
        for (int j = 0; j < 4 && col + j < N; ++j) e[j] = src[j];
    }
    return make_float4(e[0], e[1], e[2], e[3]);
}

// Four bias values for columns col .. col+3 (0 beyond N or without a bias).
__device__ __forceinline__ float4 load_bias4(const float *bias, int col, int N) {
    if (!bias) return make_float4(0.f, 0.f, 0.f, 0.f);
    if (col + 4 <= N) return *reinterpret_cast<const float4 *>(bias + col);
    float e[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < 4 && col + j < N; ++j) e[j] = bias[j + col];
    return make_float4(e[0], e[1], e[2], e[3]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Stream-K flags: a release store of the launch's epoch after a partial is
// written, and a bounded acquire spin for it on the reader's side.
__device__ __forceinline__ void publish_flag(unsigned int *flag, unsigned int epoch) {
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(epoch) : "memory");
}

__device__ __forceinline__ bool wait_flag(const unsigned int *flag, unsigned int epoch, volatile int *abort_flag,
                                          unsigned long long timeout_ns) {
    auto seen = [&]() {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        return v == epoch;
    };
    if (seen()) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (seen()) return true;
        if ((i & 31u) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                atomicOr(&g_fault_word, SITE_FIXUP);
                return false;
            }
        }
    }
}

// The GEMM kernel, one instantiation per variant (see kernel_config.h).
//   CG = 1: one CTA per 128 x BN tile.
//   CG = 2: a cluster of two CTAs per 256 x BN tile.  Both CTAs' producers
//     load their own A rows and half of B into their own rings and complete
//     on the leader's (rank 0) full barriers; the leader's MMA thread issues
//     cta_group::2 MMAs that read both CTAs' shared memory and write both
//     CTAs' tensor memory, and its commits arrive on the barriers of both
//     CTAs; each CTA's epilogue drains its own 128 rows and tells the leader
//     when its half of an accumulator is free.
template <int CG, int BN, int TK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_out,
                     const __grid_constant__ KernelParams p) {
    constexpr VariantInfo V = make_variant(CG, BN, TK);
    // Operand boxes.  K-major (A row-major, B column-major): TK/64 boxes of
    // rows x 64 K, each rows x 128 bytes.  MN-major (A column-major, B
    // row-major): rows/64 boxes of 64 M/N x TK, each TK rows of 128 bytes.
    // The stage holds the same bytes either way.
    constexpr int A_BOX = CTA_ROWS * TILE_K * 2;    // bytes of one K-major A box (128 rows x 128 bytes)
    constexpr int B_BOX = V.b_rows * TILE_K * 2;    // bytes of one K-major B box
    constexpr int MN_BOX = TK * TILE_K * 2;         // bytes of one MN-major box (TK rows x 128 bytes)
    constexpr int STAGES = V.stages;
    constexpr int BAR_FULL = 0;                           // [STAGES] operands landed (leader's count both CTAs)
    constexpr int BAR_EMPTY = STAGES;                     // [STAGES] slot free again
    constexpr int BAR_ACC_FULL = 2 * STAGES;              // [ACC_BUFS] accumulator complete
    constexpr int BAR_ACC_EMPTY = 2 * STAGES + ACC_BUFS;  // [ACC_BUFS] accumulator drained (leader's)
    constexpr int BAR_DRAIN = 2 * STAGES + 2 * ACC_BUFS;  // all MMAs of this CTA done
    constexpr int BAR_CLOAD = 2 * STAGES + 2 * ACC_BUFS + 1;   // [2 per epilogue warp] previous C landed
    constexpr int NUM_BARRIERS = 2 * STAGES + 2 * ACC_BUFS + 1 + 2 * EPI_WARPS;
    static_assert(NUM_BARRIERS_FIXED == 2 * ACC_BUFS + 1 + 2 * EPI_WARPS, "barrier count");
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(CTA_ROWS * CG, BN);
    constexpr uint32_t TX_BYTES = CG * V.stage;           // bytes both CTAs land per stage
    constexpr bool PAIR = CG == 2;

    extern __shared__ uint8_t smem_raw[];
    // Operand tiles must start on the 1024-byte swizzle-atom boundary.  The
    // layout is identical in both CTAs of a pair: the pair MMA reads the peer's
    // operands at the leader's offsets.
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sA = ptx::smem_addr(smem);                      // STAGES A tiles
    const uint32_t sB = sA + STAGES * V.a_stage;                   // STAGES B tiles
    const uint32_t sEpi = sA + STAGES * V.stage;                   // epilogue staging (1024-aligned)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * V.stage + EPI_STAGING_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARRIERS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto bar = [bar0](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const long long cluster = blockIdx.x / CG;
    const bool a_mn = p.a_mn != 0, b_mn = p.b_mn != 0;
    // Box j of an operand of `rows` rows per CTA starting at row0, in k-tile kc:
    // its tensor-map coordinates (inner first) and its offset in the stage.
    constexpr int K_BOXES = V.k_boxes;
    auto box_count = [](bool mn, int rows) { return mn ? rows / TILE_K : K_BOXES; };
    auto box_x = [](bool mn, int j, int kc, int row0) { return mn ? row0 + j * TILE_K : kc + j * TILE_K; };
    auto box_y = [](bool mn, int j, int kc, int row0) { return mn ? kc : row0; };
    auto box_off = [](bool mn, int j, int rows) { return static_cast<uint32_t>(j * (mn ? MN_BOX : rows * TILE_K * 2)); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);    // leader's producer arrive + both CTAs' bytes
            ptx::mbar_init(bar(BAR_EMPTY + s), 1);   // MMA commit
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            ptx::mbar_init(bar(BAR_ACC_FULL + b), 1);              // MMA commit
            ptx::mbar_init(bar(BAR_ACC_EMPTY + b), EPI_WARPS * CG); // one lane per epilogue warp of each CTA
        }
        ptx::mbar_init(bar(BAR_DRAIN), 1);
        for (int i = 0; i < 2 * EPI_WARPS; ++i) ptx::mbar_init(bar(BAR_CLOAD + i), 1);   // lane 0 + the box's bytes
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_a);
        ptx::prefetch_tensormap(&tmap_b);
        ptx::prefetch_tensormap(&tmap_c);
        ptx::prefetch_tensormap(&tmap_out);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), V.tmem_cols);
            ptx::tmem_relinquish_alloc_permit_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(tmem_slot), V.tmem_cols);
            ptx::tmem_relinquish_alloc_permit();
        }
    }
    ptx::tc_fence_before_sync();
    if constexpr (PAIR) {
        ptx::cluster_sync();   // both CTAs' barriers initialised and TMEM allocated
    } else {
        __syncthreads();
    }
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    // Everything above overlaps the tail of the previous kernel in the stream;
    // no global memory (operands, C, workspace, flags) is read or written
    // before it has finished.  The producer only asks L2 to start fetching
    // the operands of its first STAGES k-tiles: L2 is the point of coherence,
    // so if the previous kernel writes them, the loads after the wait still
    // see its data.
    if (warp == 0 && lane == 0 && !p.conv) {
        Schedule first(p, cluster);
        Unit w0;
        if (first.next(p, w0)) {
            const int row_a = w0.tm * V.tile_m + static_cast<int>(rank) * CTA_ROWS;
            const int row_b = w0.tn * BN + static_cast<int>(rank) * V.b_rows;
            for (int kb = 0; kb < w0.kb_count && kb < STAGES; ++kb) {
                const int kc = (w0.kb_begin + kb) * TK;
                for (int j = 0; j < box_count(a_mn, CTA_ROWS); ++j)
                    ptx::tma_prefetch_l2_2d(&tmap_a, box_x(a_mn, j, kc, row_a), box_y(a_mn, j, kc, row_a));
                for (int j = 0; j < box_count(b_mn, V.b_rows); ++j)
                    ptx::tma_prefetch_l2_2d(&tmap_b, box_x(b_mn, j, kc, row_b), box_y(b_mn, j, kc, row_b));
            }
        }
    }
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    if (warp == 0) {
        // ---------------- producer: TMA copies into the ring ----------------
        if (lane == 0) {
            uint32_t it = 0, issued = 0;
            bool ok = true;
            Schedule sched(p, cluster);
            Unit w;
            while (ok && sched.next(p, w)) {
                const int row_a = w.tm * V.tile_m + static_cast<int>(rank) * CTA_ROWS;
                const int row_b = w.tn * BN + static_cast<int>(rank) * V.b_rows;
                // convolution: the window origin of this CTA's first output pixel,
                // and the (tap, channel block) of the unit's first box -- stepped
                // box by box below, so the loop itself divides nothing
                int cv_n = 0, cv_h = 0, cv_w = 0;
                int cv_tap = 0, cv_cb = 0, cv_r = 0, cv_s = 0;
                if (p.conv) {
                    cv_n = row_a / p.cv_PQ;
                    const int pq = row_a - cv_n * p.cv_PQ;
                    const int pp = pq / p.cv_Q;
                    cv_h = pp * p.str_h - p.pad_h;
                    cv_w = (pq - pp * p.cv_Q) * p.str_w - p.pad_w;
                    const int bi0 = w.kb_begin * V.k_boxes;
                    cv_tap = bi0 / p.ncb;
                    cv_cb = bi0 - cv_tap * p.ncb;
                    cv_r = cv_tap / p.cv_S;
                    cv_s = cv_tap - cv_r * p.cv_S;
                }
                for (int kb = 0; kb < w.kb_count; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_phase<PAIR>(bar(BAR_EMPTY + s), ph ^ 1u, abort_flag, p.timeout_ns, SITE_PRODUCER,
                                          true)) {
                        ok = false;
                        break;
                    }
                    ++issued;
                    if (p.skip_load != 0 && blockIdx.x == 0 && issued == static_cast<uint32_t>(p.skip_load)) {
                        continue;   // test hook: this slot is never filled
                    }
                    if (leader) ptx::mbar_arrive_expect_tx(bar(BAR_FULL + s), TX_BYTES);
                    const int kc = (w.kb_begin + kb) * TK;
                    // the full barrier of the stage: the leader's, for both CTAs of a pair
                    const uint32_t full = PAIR ? ptx::mapa_shared(bar(BAR_FULL + s), 0) : bar(BAR_FULL + s);
                    auto load = [&](const CUtensorMap *map, uint32_t dst, int x, int y) {
                        if constexpr (PAIR) {
                            ptx::tma_load_2d_pair(dst, map, full, x, y);
                        } else {
                            ptx::tma_load_2d(dst, map, full, x, y);
                        }
                    };
                    if (p.conv) {
                        // box j: 128 pixels x 64 channels of x at one filter tap
                        // (im2col), and the matching 64 channels of that tap of
                        // the filter.  Boxes past the last tap point at channel
                        // 64 ncb (>= C): both read as zeros.
                        for (int j = 0; j < V.k_boxes; ++j) {
                            // box (kb_begin + kb) * k_boxes + j is channel block
                            // cv_cb of tap cv_tap = cv_r * S + cv_s
                            int tap = cv_tap, c0 = cv_cb * TILE_K, r = cv_r, sx = cv_s;
                            if (tap >= p.cv_taps) {
                                tap = 0;
                                c0 = p.ncb * TILE_K;
                                r = 0;
                                sx = 0;
                            }
                            if (++cv_cb == p.ncb) {
                                cv_cb = 0;
                                ++cv_tap;
                                if (++cv_s == p.cv_S) {
                                    cv_s = 0;
                                    ++cv_r;
                                }
                            }
                            const uint16_t off_h = static_cast<uint16_t>(r * p.dil_h);
                            const uint16_t off_w = static_cast<uint16_t>(sx * p.dil_w);
                            const uint32_t dst_a = sA + s * V.a_stage + j * A_BOX;
                            const uint32_t dst_b = sB + s * V.b_stage + j * B_BOX;
                            if constexpr (PAIR) {
                                ptx::tma_load_im2col_4d_pair(dst_a, &tmap_a, full, c0, cv_w, cv_h, cv_n, off_w, off_h);
                                ptx::tma_load_3d_pair(dst_b, &tmap_b, full, c0, tap, row_b);
                            } else {
                                ptx::tma_load_im2col_4d(dst_a, &tmap_a, full, c0, cv_w, cv_h, cv_n, off_w, off_h);
                                ptx::tma_load_3d(dst_b, &tmap_b, full, c0, tap, row_b);
                            }
                        }
                        continue;
                    }
                    const int na = box_count(a_mn, CTA_ROWS), nb = box_count(b_mn, V.b_rows);
                    for (int j = 0; j < na || j < nb; ++j) {
                        if (j < na)
                            load(&tmap_a, sA + s * V.a_stage + box_off(a_mn, j, CTA_ROWS), box_x(a_mn, j, kc, row_a),
                                 box_y(a_mn, j, kc, row_a));
                        if (j < nb)
                            load(&tmap_b, sB + s * V.b_stage + box_off(b_mn, j, V.b_rows), box_x(b_mn, j, kc, row_b),
                                 box_y(b_mn, j, kc, row_b));
                    }
                }
            }
            // No copy may still be writing a CTA's shared memory when it exits:
            // the leader waits (bounded) for the last STAGES stages, whose full
            // barriers count both CTAs' bytes; the peer cannot pass the final
            // cluster barrier before the leader does.  Earlier stages were
            // consumed by the MMA thread before their slots were reused.
            if (leader) {
                const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
                for (uint32_t j = first; j < it; ++j) {
                    wait_phase<PAIR>(bar(BAR_FULL + j % STAGES), (j / STAGES) & 1u, abort_flag, p.timeout_ns,
                                     SITE_DRAIN, false);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: one thread of the leader CTA ------------
        if (lane == 0 && leader) {
            uint32_t it = 0, tc = 0;
            bool ok = true;
            Schedule sched(p, cluster);
            Unit w;
            for (; ok && sched.next(p, w); ++tc) {
                const uint32_t buf = tc & 1u;
                const uint32_t use = tc >> 1;
                if (!wait_phase<PAIR>(bar(BAR_ACC_EMPTY + buf), (use & 1u) ^ 1u, abort_flag, p.timeout_ns,
                                      SITE_MMA_ACC, true)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * BN;
                const uint32_t idesc = IDESC | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
                for (int kb = 0; kb < w.kb_count; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_phase<PAIR>(bar(BAR_FULL + s), ph, abort_flag, p.timeout_ns, SITE_MMA_OPERANDS, true)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int k = 0; k < TK / MMA_K; ++k) {
                        // K-major: box k/4 of the k-tile; inside it, the next 16
                        // elements of K are +32 bytes in the swizzled 128-byte
                        // row, i.e. +2 in the address>>4 field of the descriptor.
                        // MN-major: 16 more rows of K, two swizzle atoms on.
                        const int j = k / (TILE_K / MMA_K);
                        const uint32_t step = 2u * static_cast<uint32_t>(k % (TILE_K / MMA_K));
                        const uint32_t a_base = sA + s * V.a_stage, b_base = sB + s * V.b_stage;
                        const uint64_t a_desc =
                            a_mn ? ptx::smem_desc_mnmajor_sw128(a_base + k * (MMA_K * 128), MN_BOX)
                                 : ptx::smem_desc_kmajor_sw128(a_base + j * A_BOX) + step;
                        const uint64_t b_desc =
                            b_mn ? ptx::smem_desc_mnmajor_sw128(b_base + k * (MMA_K * 128), MN_BOX)
                                 : ptx::smem_desc_kmajor_sw128(b_base + j * B_BOX) + step;
                        const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
                        if constexpr (PAIR) {
                            ptx::mma_bf16_pair(d_tmem, a_desc, b_desc, idesc, acc);
                        } else {
                            ptx::mma_bf16(d_tmem, a_desc, b_desc, idesc, acc);
                        }
                    }
                    // slot reusable (in every CTA) once these MMAs have read it
                    if constexpr (PAIR) {
                        ptx::mma_commit_pair_multicast(bar(BAR_EMPTY + s), 0x3);
                    } else {
                        ptx::mma_commit(bar(BAR_EMPTY + s));
                    }
                }
                if (!ok) break;
                // accumulator complete (in every CTA)
                if constexpr (PAIR) {
                    ptx::mma_commit_pair_multicast(bar(BAR_ACC_FULL + buf), 0x3);
                } else {
                    ptx::mma_commit(bar(BAR_ACC_FULL + buf));
                }
            }
            // Every MMA issued here must finish before TMEM is released.
            if constexpr (PAIR) {
                ptx::mma_commit_pair(bar(BAR_DRAIN));
            } else {
                ptx::mma_commit(bar(BAR_DRAIN));
            }
            wait_phase<PAIR>(bar(BAR_DRAIN), 0, abort_flag, p.timeout_ns, SITE_DRAIN, false);
        }
    } else {
        // ---------------- epilogue: TMEM -> registers -> global ---------------
        const int quarter = warp & 3;            // TMEM lanes this warp may read: 32*quarter ..
        // This warp's two staging buffers for TMA stores of C.  A 32 x 32 chunk
        // is staged row per lane, with the 16-byte pieces of each row permuted
        // the way the tensor map's swizzle reads them (bf16: 64-byte rows,
        // piece ^ ((row >> 1) & 3); fp32: 128-byte rows, piece ^ (row & 7)),
        // which also keeps the 32 lanes' writes free of bank conflicts.
        const uint32_t epi_buf0 = sEpi + static_cast<uint32_t>(quarter) * 2u * EPI_BUF_BYTES;
        uint32_t stores_issued = 0;
        uint32_t c_phase = 0;     // bit b: parity of the next completion of this warp's C-load barrier b
        uint32_t c_pending = 0;   // bit b: a load of previous C into buffer b not yet waited for
        uint32_t tc = 0;
        Schedule sched(p, cluster);
        Unit w;
        for (; sched.next(p, w); ++tc) {
            const uint32_t buf = tc & 1u;
            const uint32_t use = tc >> 1;
            const bool ok =
                wait_phase<PAIR>(bar(BAR_ACC_FULL + buf), use & 1u, abort_flag, p.timeout_ns, SITE_EPI_ACC, true);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN;
            const int col_base = w.tn * BN;
            const int flag_idx = static_cast<int>(rank) * EPI_WARPS + quarter;   // within a slot
            // Stream-K owner: the other segments of this tile are the first
            // units of the next clusters whose ranges start inside the tile;
            // wait until each has published its partial for these 32 rows.
            long long contrib_end = cluster + 1;
            if (w.kind == KIND_OWNER) {
                const long long tile_end = static_cast<long long>(w.sk_tile + 1) * p.k_tiles;
                while (contrib_end < p.num_clusters && sk_range_start(p, contrib_end) < tile_end) ++contrib_end;
                bool got = true;
                for (long long c2 = cluster + 1; c2 < contrib_end && got; ++c2) {
                    if (sk_range_start(p, c2 + 1) == sk_range_start(p, c2)) continue;   // empty range: no partial
                    got = wait_flag(p.sk_flags + c2 * (CG * EPI_WARPS) + flag_idx, p.epoch, abort_flag,
                                    p.timeout_ns);
                }
            }
            // A partial slot holds a tile in warp-major order: for each
            // (CTA, warp quarter, 32-column chunk, float4 v), the 32 lanes' float4s
            // are consecutive, so every warp access moves 512 contiguous bytes.
            // Lane l of the warp at (rank, quarter) owns row quarter*32 + l.
            const long long slot_floats = static_cast<long long>(V.tile_m) * BN;
            const int warp_chunk0 = (static_cast<int>(rank) * EPI_WARPS + quarter) * (BN / 32);
            auto slot_ptr = [&](long long slot, int chunk) {
                return reinterpret_cast<float4 *>(p.partials + slot * slot_floats) +
                       (static_cast<long long>(warp_chunk0 + chunk) * 8) * 32 + lane;
            };
            // where this unit's partial tile goes: its split-K slot, or (stream-K)
            // this cluster's slot
            const bool to_slot = w.kind == KIND_PARTIAL || p.split_k > 1;
            const long long my_slot =
                p.split_k > 1 ? static_cast<long long>(w.split) * p.tiles_m * p.tiles_n +
                                    static_cast<long long>(w.tm) * p.tiles_n + w.tn
                              : cluster;
            // stream-K owner: partial sums of the first contributor, one chunk ahead
            float4 pre[8];
            auto prefetch = [&](int chunk) {
                const float4 *src = slot_ptr(cluster + 1, chunk);
#pragma unroll
                for (int v = 0; v < 8; ++v) pre[v] = __ldcg(src + v * 32);
            };
            const bool owner_fast = w.kind == KIND_OWNER && contrib_end == cluster + 2;   // the common case
            // chunks this warp handles: all of them for a partial tile, else
            // those that start inside C (the same for the whole warp)
            const int n_chunks = to_slot ? BN / 32 : min(BN / 32, (p.N - col_base + 31) / 32);
            const int warp_row0 = w.tm * V.tile_m + static_cast<int>(rank) * CTA_ROWS + quarter * 32;
            // stream-K owner: add the later segments of chunk c in k order
            auto add_partials = [&](uint32_t (&r)[32], int c) {
                for (long long c2 = cluster + 1; c2 < contrib_end; ++c2) {
                    if (sk_range_start(p, c2 + 1) == sk_range_start(p, c2)) continue;
                    const float4 *src = slot_ptr(c2, c);
                    float4 q[8];
#pragma unroll
                    for (int v = 0; v < 8; ++v) q[v] = __ldcg(src + v * 32);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + q[v].x);
                        r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + q[v].y);
                        r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + q[v].z);
                        r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + q[v].w);
                    }
                }
            };
            // stage the chunk and hand it to TMA, which clips rows >= M and
            // columns >= N
            auto stage_store = [&](uint32_t (&r)[32], int col0) {
                if (warp_row0 >= p.M) return;
                if (stores_issued >= 2 && lane == 0) ptx::bulk_wait_group_read<1>();   // this buffer read out
                __syncwarp();
                const uint32_t buf = epi_buf0 + (stores_issued & 1u) * EPI_BUF_BYTES;
                if (p.out_bf16) {
                    const uint32_t row_base = buf + static_cast<uint32_t>(lane) * 64u;
                    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        ptx::st_shared_v4(row_base + ((static_cast<uint32_t>(v) ^ sw) << 4),
                                          pack_bf16x2(r[8 * v + 0], r[8 * v + 1]), pack_bf16x2(r[8 * v + 2], r[8 * v + 3]),
                                          pack_bf16x2(r[8 * v + 4], r[8 * v + 5]), pack_bf16x2(r[8 * v + 6], r[8 * v + 7]));
                    }
                } else {
                    const uint32_t row_base = buf + static_cast<uint32_t>(lane) * 128u;
                    const uint32_t sw = static_cast<uint32_t>(lane) & 7u;
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        ptx::st_shared_v4(row_base + ((static_cast<uint32_t>(v) ^ sw) << 4), r[4 * v + 0], r[4 * v + 1],
                                          r[4 * v + 2], r[4 * v + 3]);
                    }
                }
                ptx::fence_proxy_async_shared();
                __syncwarp();
                // Every chunk commits a bulk group, empty when the chunk lies
                // wholly past n_tma, so that buffers and groups keep in step.
                if (lane == 0) {
                    if (col0 < p.n_tma) ptx::tma_store_2d(&tmap_out, buf, col0, warp_row0);
                    ptx::bulk_commit_group();
                }
                ++stores_issued;
            };
            // The fused path's results go from registers straight to C: each lane
            // writes its own row's 32 values with 16-byte stores (a row of C
            // starts on a 16-byte boundary, ldc being a whole number of 16-byte
            // pieces), which keeps them off shared memory, busy with the main
            // loop's operands.  Columns past N are not written.
            auto direct_store = [&](uint32_t (&r)[32], int col0) {
                const int row = warp_row0 + lane;
                if (row >= p.M) return;
                const long long at = static_cast<long long>(row) * p.ld_out + col0;
                if (p.out_bf16) {
                    uint16_t *dst = static_cast<uint16_t *>(p.out) + at;
                    if (col0 + 32 <= p.N) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            *reinterpret_cast<uint4 *>(dst + 8 * v) =
                                make_uint4(pack_bf16x2(r[8 * v + 0], r[8 * v + 1]), pack_bf16x2(r[8 * v + 2], r[8 * v + 3]),
                                           pack_bf16x2(r[8 * v + 4], r[8 * v + 5]), pack_bf16x2(r[8 * v + 6], r[8 * v + 7]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < p.N) dst[j] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[j])));
                    }
                } else {
                    uint32_t *dst = static_cast<uint32_t *>(p.out) + at;
                    if (col0 + 32 <= p.N) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            *reinterpret_cast<uint4 *>(dst + 4 * v) = make_uint4(r[4 * v + 0], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < p.N) dst[j] = r[j];
                    }
                }
            };
            bool c_ok = true;   // false: a wait for previous C gave up (the CTA aborts)
            if (p.epi && !to_slot) {
                // Fused epilogue, one chunk at a time in a rolled loop so that the
                // code stays small (the epilogue warps share the instruction
                // cache with the producer and MMA threads).  The linear part and
                // the activation run on the chunk's 32 registers, two values per
                // paired instruction, with no round trip through shared memory,
                // whose bandwidth the main loop's copies and MMAs are using.
                // With beta != 0 the previous C comes in by TMA, one 32 x 32 chunk
                // ahead, into the warp's two staging buffers (no store leaves
                // from them in a fused launch), in the swizzled layout of a store
                // (rows past M and columns past N arrive as zeros); each lane then
                // reads its own row of it.  Chunk c lands in buffer c & 1.
                const bool read_c = p.beta != 0.0f && warp_row0 < p.M;   // warp-uniform
                const uint32_t c_bar = bar(BAR_CLOAD + 2 * quarter);
                const uint32_t c_bytes = 32u * 32u * (p.out_bf16 ? 2u : 4u);
                auto load_c_chunk = [&](int col0, uint32_t slot) {
                    c_pending |= 1u << slot;
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(c_bar + 8u * slot, c_bytes);
                        ptx::tma_load_2d(epi_buf0 + slot * EPI_BUF_BYTES, &tmap_c, c_bar + 8u * slot, col0, warp_row0);
                    }
                };
                if (read_c) {
                    __syncwarp();   // the previous unit's reads of buffer 0 are done
                    load_c_chunk(col_base, 0u);
                }
                if (owner_fast) prefetch(0);
                const uint64_t alpha2 = ptx::f2_splat(p.alpha), beta2 = ptx::f2_splat(p.beta);
                // A chunk's 32 bias values are the same for every lane: eight
                // 16-byte loads of one address per warp (bias is 16-byte aligned).
                // The next chunk's go out as soon as this chunk's linear part has
                // used them, and land during its activation and store.  Columns
                // past N read as 0.
                float4 bq[8];
                auto load_bias = [&](int col0) {
                    if (p.bias == nullptr) {
#pragma unroll
                        for (int v = 0; v < 8; ++v) bq[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else if (col0 + 32 <= p.N) {
#pragma unroll
                        for (int v = 0; v < 8; ++v) bq[v] = __ldg(reinterpret_cast<const float4 *>(p.bias + col0) + v);
                    } else {
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const int j = col0 + 4 * v;
                            bq[v] = make_float4(j < p.N ? __ldg(p.bias + j) : 0.f, j + 1 < p.N ? __ldg(p.bias + j + 1) : 0.f,
                                                j + 2 < p.N ? __ldg(p.bias + j + 2) : 0.f,
                                                j + 3 < p.N ? __ldg(p.bias + j + 3) : 0.f);
                        }
                    }
                };
                load_bias(col_base);
#pragma unroll 1
                for (int c = 0; c < n_chunks; ++c) {
                    const int col0 = col_base + c * 32;
                    const uint32_t slot = static_cast<uint32_t>(c) & 1u;
                    // previous C of this lane's row, as 16 pairs of fp32 bit patterns
                    uint64_t cp[16];
                    if (read_c) {
                        if (c + 1 < n_chunks) {
                            // every lane has used the previous chunk's C: the next
                            // chunk's lands in its buffer
                            __syncwarp();
                            load_c_chunk(col0 + 32, slot ^ 1u);
                        }
                        c_ok = __all_sync(0xffffffffu, wait_phase<false>(c_bar + 8u * slot, (c_phase >> slot) & 1u,
                                                                         abort_flag, p.timeout_ns, SITE_EPI_C, true));
                        if (!c_ok) {
                            // loads may still be landing in the buffers: wait for them
                            // (bounded) before this warp leaves
                            for (uint32_t b = 0; b < 2; ++b)
                                if ((c_pending >> b) & 1u)
                                    wait_phase<false>(c_bar + 8u * b, (c_phase >> b) & 1u, abort_flag, p.timeout_ns,
                                                      SITE_EPI_C, false);
                            break;
                        }
                        c_phase ^= 1u << slot;
                        c_pending &= ~(1u << slot);
                        const uint32_t cbuf = epi_buf0 + slot * EPI_BUF_BYTES;
                        if (p.out_bf16) {
                            // a bf16 is the high half of the fp32 with the same value
                            const uint32_t row_base = cbuf + static_cast<uint32_t>(lane) * 64u;
                            const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const uint4 u = ptx::ld_shared_v4(row_base + ((static_cast<uint32_t>(v) ^ sw) << 4));
                                cp[4 * v + 0] = ptx::f2_pack(u.x << 16, u.x & 0xFFFF0000u);
                                cp[4 * v + 1] = ptx::f2_pack(u.y << 16, u.y & 0xFFFF0000u);
                                cp[4 * v + 2] = ptx::f2_pack(u.z << 16, u.z & 0xFFFF0000u);
                                cp[4 * v + 3] = ptx::f2_pack(u.w << 16, u.w & 0xFFFF0000u);
                            }
                        } else {
                            const uint32_t row_base = cbuf + static_cast<uint32_t>(lane) * 128u;
                            const uint32_t sw = static_cast<uint32_t>(lane) & 7u;
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const uint4 u = ptx::ld_shared_v4(row_base + ((static_cast<uint32_t>(v) ^ sw) << 4));
                                cp[2 * v + 0] = ptx::f2_pack(u.x, u.y);
                                cp[2 * v + 1] = ptx::f2_pack(u.z, u.w);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) cp[j] = 0;
                    }
                    uint32_t r[32];
                    __syncwarp();
                    ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
                    ptx::tmem_wait_ld(r);
                    if (owner_fast) {
                        // the contributor's partial sums of this chunk, loaded a
                        // chunk ahead; the next chunk's go out now and land while
                        // this one is finished and stored
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + pre[v].x);
                            r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + pre[v].y);
                            r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + pre[v].z);
                            r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + pre[v].w);
                        }
                        if (c + 1 < n_chunks) prefetch(c + 1);
                    } else if (w.kind == KIND_OWNER) {
                        add_partials(r, c);
                    }
                    // alpha * acc + beta * c + bias, each product and sum rounded
                    // on its own, as epilogue_linear does
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        uint64_t lo = ptx::f2_mul(alpha2, ptx::f2_pack(r[4 * v + 0], r[4 * v + 1]));
                        uint64_t hi = ptx::f2_mul(alpha2, ptx::f2_pack(r[4 * v + 2], r[4 * v + 3]));
                        lo = ptx::f2_add(lo, ptx::f2_mul(beta2, cp[2 * v + 0]));
                        hi = ptx::f2_add(hi, ptx::f2_mul(beta2, cp[2 * v + 1]));
                        lo = ptx::f2_add(lo, ptx::f2_pack(__float_as_uint(bq[v].x), __float_as_uint(bq[v].y)));
                        hi = ptx::f2_add(hi, ptx::f2_pack(__float_as_uint(bq[v].z), __float_as_uint(bq[v].w)));
                        ptx::f2_unpack(lo, r[4 * v + 0], r[4 * v + 1]);
                        ptx::f2_unpack(hi, r[4 * v + 2], r[4 * v + 3]);
                    }
                    if (c + 1 < n_chunks) load_bias(col0 + 32);
                    if (p.act == GEMM_ACT_GELU) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint64_t y = gelu2(ptx::f2_pack(r[2 * j], r[2 * j + 1]));
                            ptx::f2_unpack(y, r[2 * j], r[2 * j + 1]);
                        }
                    }
                    if (p.act == GEMM_ACT_RELU) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(fmaxf(__uint_as_float(r[q]), 0.0f));
                    }
                    direct_store(r, col0);
                }
            } else {
            if (owner_fast) prefetch(0);
            // Two register sets: chunk c+1 is read from TMEM while chunk c is
            // converted and stored.
            uint32_t rbuf[2][32];
            __syncwarp();
            ptx::tmem_ld_32x32b_x32(t_row, rbuf[0]);
            ptx::tmem_wait_ld(rbuf[0]);
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                if (c >= n_chunks) break;
                const int col0 = col_base + c * 32;
                uint32_t (&r)[32] = rbuf[c & 1];
                if (c + 1 < n_chunks) {
                    __syncwarp();
                    ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>((c + 1) * 32), rbuf[(c + 1) & 1]);
                }
                if (to_slot) {
                    // the whole tile-row chunk, in range or not: a reader takes it back
                    float4 *dst = slot_ptr(my_slot, c);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        __stcg(dst + v * 32, make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                                         __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
                    }
                    if (c + 1 < n_chunks) ptx::tmem_wait_ld(rbuf[(c + 1) & 1]);
                    continue;
                }
                if (w.kind == KIND_OWNER) {
                    if (owner_fast) {
                        // the first (usually only) contributor's partial sums, one chunk ahead
                        float4 q[8];
#pragma unroll
                        for (int v = 0; v < 8; ++v) q[v] = pre[v];
                        if (c + 1 < BN / 32 && col0 + 32 < p.N) prefetch(c + 1);
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + q[v].x);
                            r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + q[v].y);
                            r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + q[v].z);
                            r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + q[v].w);
                        }
                    } else {
                        add_partials(r, c);
                    }
                }
                stage_store(r, col0);
                if (c + 1 < n_chunks) ptx::tmem_wait_ld(rbuf[(c + 1) & 1]);
            }
            }
            if (!c_ok) break;
            if (!to_slot && !p.epi && warp_row0 < p.M && col_base + n_chunks * 32 > p.n_tma) {
                // C's columns from n_tma to N, when N is not a whole number of
                // 16-byte pieces: a TMA store clipped at N would still write
                // the last piece whole, past N.  They lie in the last chunk,
                // still in its staging buffer; each lane stores its own row's.
                const int col0 = col_base + (n_chunks - 1) * 32;
                const uint32_t sbuf = epi_buf0 + ((stores_issued - 1u) & 1u) * EPI_BUF_BYTES;
                const int row = warp_row0 + lane;
                if (row < p.M) {
                    const long long at = static_cast<long long>(row) * p.ld_out + col0;
                    const int j1 = min(p.N - col0, 32);
                    for (int j = max(p.n_tma - col0, 0); j < j1; ++j) {
                        const uint32_t uj = static_cast<uint32_t>(j);
                        if (p.out_bf16) {
                            const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
                            static_cast<uint16_t *>(p.out)[at + j] = ptx::ld_shared_b16(
                                sbuf + static_cast<uint32_t>(lane) * 64u + (((uj >> 3) ^ sw) << 4) + (uj & 7u) * 2u);
                        } else {
                            const uint32_t sw = static_cast<uint32_t>(lane) & 7u;
                            static_cast<uint32_t *>(p.out)[at + j] = ptx::ld_shared_b32(
                                sbuf + static_cast<uint32_t>(lane) * 128u + (((uj >> 2) ^ sw) << 4) + (uj & 3u) * 4u);
                        }
                    }
                }
            }
            if (w.kind == KIND_OWNER && lane == 0) {
                // The owner clears the flags it consumed, so that every launch
                // starts from cleared flags -- also one replayed from a captured
                // graph, which carries the epoch it was captured with.  (The next
                // launch in the stream writes flags only after this grid ends.)
                for (long long c2 = cluster + 1; c2 < contrib_end; ++c2)
                    if (sk_range_start(p, c2 + 1) != sk_range_start(p, c2))
                        p.sk_flags[c2 * (CG * EPI_WARPS) + flag_idx] = 0u;
            }
            if (w.kind == KIND_PARTIAL) {
                // publish: every lane's stores, then one release of the flag
                __threadfence();
                __syncwarp();
                if (lane == 0) publish_flag(p.sk_flags + cluster * (CG * EPI_WARPS) + flag_idx, p.epoch);
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) {
                    ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(BAR_ACC_EMPTY + buf), 0));
                } else {
                    ptx::mbar_arrive(bar(BAR_ACC_EMPTY + buf));
                }
            }
        }
    }

    if (warp >= 2 && lane == 0) ptx::bulk_wait_group_all();   // C written before the CTA ends
    __syncwarp();
    ptx::tc_fence_before_sync();
    if constexpr (PAIR) {
        ptx::cluster_sync();   // no CTA leaves while its peer may still touch its memory
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        if constexpr (PAIR) {
            ptx::tmem_dealloc_pair(tmem_base, V.tmem_cols);
        } else {
            ptx::tmem_dealloc(tmem_base, V.tmem_cols);
        }
    }
}

// C[m][n] = the sum over the split slices s = 0 .. split-1 of slice s's
// partial tile, in a fixed order, then cast to the output type.  Partial
// slots are warp-major (as the GEMM epilogue writes them): float4 q of a slot
// holds row wq*32 + lane, columns chunk*32 + 4v .. +3, where
// q = ((wq*(bn/32) + chunk)*8 + v)*32 + lane.
// A CTA of 8 warps takes 32 consecutive float4s of the slots (one per lane);
// warp w adds slices w, w+8, w+16, ... in increasing order (BATCH loads in
// flight: the smallest of 2, 4, 8, 16, 24 that covers a warp's slices, else
// 24 per round), and warp 0 then adds the 8 warp sums in order w = 0 .. 7.  The
// order is the same on every run, whatever BATCH.
// With the fused epilogue (ep.epi), the sum of the slices takes the place of
// the accumulator: C := act(alpha * sum + beta * C + bias[n]).
constexpr int COMBINE_WARPS = 8;

struct EpilogueArgs {
    int epi;
    float alpha, beta;
    const float *bias;
    int act;
};

// Small batches keep to 64 registers (4 CTAs per SM), so that with a few
// slices the whole grid fits on the SMs the GEMM leaves idle and waits there
// (programmatic dependent launch); large ones take 128 (2 CTAs per SM) to
// hold all their loads in flight.
template <int BATCH>
__global__ void __launch_bounds__(COMBINE_WARPS * 32, BATCH <= 8 ? 4 : 2)
    splitk_combine_kernel(const float *__restrict__ part, int split, long long tiles, int tiles_n, int tile_m, int bn,
                          int M, int N, void *C, long long ldc, int out_bf16, EpilogueArgs ep) {
    __shared__ float4 warp_sum[COMBINE_WARPS][32];
    ptx::grid_dependency_wait();   // the partials come from the previous kernel in the stream
    ptx::grid_launch_dependents();
    const long long slot_f4 = static_cast<long long>(tile_m) * bn / 4;
    const long long split_f4 = tiles * slot_f4;
    const int chunks = bn / 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const float4 *P = reinterpret_cast<const float4 *>(part);
    for (long long base = blockIdx.x * 32LL; base < split_f4; base += gridDim.x * 32LL) {
        const long long idx = base + lane;
        // where this float4 lands in C
        const long long tile = idx / slot_f4;
        const int q = static_cast<int>(idx - tile * slot_f4);
        const int v = (q >> 5) & 7;
        const int chunk = (q >> 8) % chunks;
        const int wq = (q >> 8) / chunks;
        const int row = static_cast<int>(tile / tiles_n) * tile_m + wq * 32 + lane;
        const int col = static_cast<int>(tile % tiles_n) * bn + chunk * 32 + v * 4;
        const bool live = idx < split_f4 && row < M && col < N;   // padding of the tiles is never read
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
            // Every load of a round is issued before the first add, the
            // round's tail included, so a warp's slices cost
            // ceil(slices / BATCH) memory round trips; the adds then
            // run in increasing slice order.
            const float4 *src = P + idx;
            for (int s = warp; s < split; s += BATCH * COMBINE_WARPS) {
                float4 w[BATCH];
#pragma unroll
                for (int j = 0; j < BATCH; ++j) {
                    // past the last slice: reload the last one (in bounds, not
                    // added), so the loads stay unconditional and all issue first
                    const int sj = min(s + j * COMBINE_WARPS, split - 1);
                    w[j] = __ldcs(src + static_cast<long long>(sj) * split_f4);
                }
                // A reloaded slice adds +0 instead, which leaves acc unchanged:
                // acc starts at +0 and a sum of finite values is -0 only when
                // both terms are -0, so acc is never -0.
#pragma unroll
                for (int j = 0; j < BATCH; ++j) {
                    const bool in = s + j * COMBINE_WARPS < split;
                    acc.x += in ? w[j].x : 0.0f;
                    acc.y += in ? w[j].y : 0.0f;
                    acc.z += in ? w[j].z : 0.0f;
                    acc.w += in ? w[j].w : 0.0f;
                }
            }
        }
        warp_sum[warp][lane] = acc;
        __syncthreads();
        if (warp == 0 && live) {
            float4 t = warp_sum[0][lane];
            for (int w2 = 1; w2 < COMBINE_WARPS && w2 < split; ++w2) {
                const float4 u = warp_sum[w2][lane];
                t.x += u.x;
                t.y += u.y;
                t.z += u.z;
                t.w += u.w;
            }
            if (ep.epi) {
                const float4 c = ep.beta != 0.0f ? load_c4(C, ldc, out_bf16, row, col, N) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 b = load_bias4(ep.bias, col, N);
                t.x = epilogue_value(t.x, c.x, b.x, ep.alpha, ep.beta, ep.act);
                t.y = epilogue_value(t.y, c.y, b.y, ep.alpha, ep.beta, ep.act);
                t.z = epilogue_value(t.z, c.z, b.z, ep.alpha, ep.beta, ep.act);
                t.w = epilogue_value(t.w, c.w, b.w, ep.alpha, ep.beta, ep.act);
            }
            {
                const float a[4] = {t.x, t.y, t.z, t.w};
                if (out_bf16) {
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(C) + static_cast<long long>(row) * ldc + col;
                    if (col + 4 <= N) {
                        const __nv_bfloat162 lo = __floats2bfloat162_rn(a[0], a[1]);
                        const __nv_bfloat162 hi = __floats2bfloat162_rn(a[2], a[3]);
                        uint2 u2;
                        u2.x = *reinterpret_cast<const uint32_t *>(&lo);
                        u2.y = *reinterpret_cast<const uint32_t *>(&hi);
                        *reinterpret_cast<uint2 *>(dst) = u2;
                    } else {
                        for (int j = 0; j < 4 && col + j < N; ++j) dst[j] = __float2bfloat16_rn(a[j]);
                    }
                } else {
                    float *dst = static_cast<float *>(C) + static_cast<long long>(row) * ldc + col;
                    if (col + 4 <= N) {
                        *reinterpret_cast<float4 *>(dst) = t;
                    } else {
                        for (int j = 0; j < 4 && col + j < N; ++j) dst[j] = a[j];
                    }
                }
            }
        }
        __syncthreads();
    }
}

// K == 0: C is the empty sum, zero.
__global__ void __launch_bounds__(256) fill_zero_kernel(void *C, long long ldc, int M, int N, int esize) {
    const long long total = static_cast<long long>(M) * N;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long m = idx / N;
        const long long n = idx - m * N;
        if (esize == 2) {
            static_cast<uint16_t *>(C)[m * ldc + n] = 0;
        } else {
            static_cast<float *>(C)[m * ldc + n] = 0.0f;
        }
    }
}

// K == 0 with the fused epilogue: the product is zero, C := act(beta * C + bias[n]).
__global__ void __launch_bounds__(256) epilogue_only_kernel(void *C, long long ldc, int M, int N, int out_bf16,
                                                            EpilogueArgs ep) {
    const long long total = static_cast<long long>(M) * N;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long m = idx / N;
        const long long n = idx - m * N;
        const float b = ep.bias ? ep.bias[n] : 0.0f;
        if (out_bf16) {
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(C) + m * ldc + n;
            const float c = ep.beta != 0.0f ? __bfloat162float(*dst) : 0.0f;
            *dst = __float2bfloat16_rn(epilogue_value(0.0f, c, b, ep.alpha, ep.beta, ep.act));
        } else {
            float *dst = static_cast<float *>(C) + m * ldc + n;
            const float c = ep.beta != 0.0f ? *dst : 0.0f;
            *dst = epilogue_value(0.0f, c, b, ep.alpha, ep.beta, ep.act);
        }
    }
}

// ------------------------------------------------------------------ host side

namespace {

constexpr int kMaxDevices = 64;

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, KernelParams);

KernelFn kernel_fn(int variant) {
    switch (variant) {
        case VARIANT_2SM_256x256: return gemm_bf16_kernel<2, 256, 128>;
        case VARIANT_2SM_256x128: return gemm_bf16_kernel<2, 128, 64>;
        case VARIANT_1SM_128x128: return gemm_bf16_kernel<1, 128, 64>;
        default: return gemm_bf16_kernel<1, 256, 64>;
    }
}

struct VariantState {
    int regs_per_thread = 0;
    int max_active_clusters = 0;   // 0 for single-CTA variants
};

constexpr int kMaxFlagSlots = 1024;   // clusters x CTAs x epilogue warps, bounds the stream-K flags

struct DeviceState {
    bool ready = false;
    gemm_device_desc_t desc{};
    VariantState var[VARIANT_COUNT];
    // The split-K / stream-K workspace and its size, guarded by ws_mutex.  A
    // launch that uses it holds ws_mutex from the size check until its
    // kernels are enqueued, so no other host thread can free the buffer in
    // between (a grower synchronises the device before freeing, which then
    // waits for those kernels).
    std::mutex ws_mutex;
    float *workspace = nullptr;
    size_t workspace_bytes = 0;
    unsigned int *sk_flags = nullptr;   // zeroed once; contributors publish the launch's epoch, owners clear
    unsigned int epoch = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
PFN_cuTensorMapEncodeIm2col_v12000 g_encode_im2col = nullptr;

gemm_status_t query_desc(int device, gemm_device_desc_t *d) {
    struct {
        cudaDeviceAttr attr;
        int *dst;
    } q[] = {
        {cudaDevAttrMultiProcessorCount, &d->num_sms},
        {cudaDevAttrMaxSharedMemoryPerMultiprocessor, &d->smem_per_sm},
        {cudaDevAttrMaxSharedMemoryPerBlockOptin, &d->smem_optin_per_cta},
        {cudaDevAttrReservedSharedMemoryPerBlock, &d->smem_reserved_per_cta},
        {cudaDevAttrMaxRegistersPerMultiprocessor, &d->regs_per_sm},
        {cudaDevAttrMaxThreadsPerMultiProcessor, &d->max_threads_per_sm},
        {cudaDevAttrMaxBlocksPerMultiprocessor, &d->max_ctas_per_sm},
    };
    for (auto &e : q) {
        if (cudaDeviceGetAttribute(e.dst, e.attr, device) != cudaSuccess) return GEMM_ERR_NO_DEVICE;
    }
    d->tmem_cols_per_sm = 512;   // sm_100-class tensor memory: 128 lanes x 512 columns of 32 bits
    return GEMM_OK;
}

cudaLaunchAttribute cluster_attr(int cluster_size) {
    cudaLaunchAttribute a{};
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = static_cast<unsigned>(cluster_size);
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    return a;
}

gemm_status_t init_variant(int variant, int num_sms, VariantState &vs) {
    const VariantInfo vi = variant_info(variant);
    KernelFn fn = kernel_fn(variant);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, vi.smem) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return GEMM_ERR_LAUNCH;
    vs.regs_per_thread = fa.numRegs;
    vs.max_active_clusters = 0;
    if (vi.cta_group > 1) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms / vi.cta_group * vi.cta_group));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = vi.smem;
        cudaLaunchAttribute attr = cluster_attr(vi.cta_group);
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(fn), &cfg) != cudaSuccess || n <= 0)
            return GEMM_ERR_LAUNCH;
        vs.max_active_clusters = n;
    }
    return GEMM_OK;
}

// Per-device one-time set-up, under g_mutex.
gemm_status_t device_state(int device, DeviceState **out) {
    if (device < 0 || device >= kMaxDevices) return GEMM_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &ds = g_devices[device];
    if (!ds.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
            return GEMM_ERR_NO_DEVICE;
        if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;   // built for sm_103a only
        gemm_status_t st = query_desc(device, &ds.desc);
        if (st != GEMM_OK) return st;
        for (int v = 1; v < VARIANT_COUNT; ++v) {
            st = init_variant(v, ds.desc.num_sms, ds.var[v]);
            if (st != GEMM_OK) {
                cudaGetLastError();
                return st;
            }
        }
        if (!g_encode_tiled) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult qr{};
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                    cudaSuccess ||
                qr != cudaDriverEntryPointSuccess || fn == nullptr)
                return GEMM_ERR_LAUNCH;
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        if (!g_encode_im2col) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult qr{};
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn, 12000, cudaEnableDefault, &qr) !=
                    cudaSuccess ||
                qr != cudaDriverEntryPointSuccess || fn == nullptr)
                return GEMM_ERR_LAUNCH;
            g_encode_im2col = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(fn);
        }
        ds.ready = true;
    }
    *out = &ds;
    return GEMM_OK;
}

gemm_kernel_desc_t kernel_desc(int variant, const VariantState &vs) {
    const VariantInfo vi = variant_info(variant);
    gemm_kernel_desc_t k{};
    k.regs_per_thread = vs.regs_per_thread;
    k.threads_per_cta = NUM_THREADS;
    k.smem_per_cta = vi.smem;
    k.tmem_cols_per_cta = vi.tmem_cols;
    k.cluster_size = vi.cta_group;
    k.max_active_clusters = vs.max_active_clusters;
    return k;
}

// A bf16 operand stored as `outer` lines of `inner` contiguous elements, `ld`
// apart, read in boxes of 64 inner elements (128 bytes, one swizzle span) x
// `box_outer` lines.  K-major operands: inner = K, lines = rows of the tile.
// MN-major operands: inner = M or N, lines = K.
gemm_status_t encode_operand(CUtensorMap *map, const void *ptr, int64_t inner, int64_t outer, int64_t ld,
                             int box_outer) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(TILE_K), static_cast<cuuint32_t>(box_outer)};
    cuuint32_t elem_strides[2] = {1, 1};
    // L2 fetches in 256-byte blocks when every line starts on a 128-byte
    // boundary: a block then also holds the next box's bytes of the line.  A
    // line pitch that is not a multiple of 128 bytes makes each 128-byte box
    // line straddle two L2 lines, and 256-byte blocks would fetch twice what
    // is read (measured at K = 4088: 102.3 us with 256-byte, 95.5 us with
    // 128-byte promotion; 76.6 against 78.3 us the other way at K = 4096).
    const CUtensorMapL2promotion promotion =
        (ld * 2) % 128 == 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                                elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promotion,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

// C (row-major, `rows` x `cols`, `ld` apart) as 32 x 32 boxes for the
// epilogue's TMA stores, swizzled as the epilogue stages them: bf16 rows are
// 64 bytes (64-byte swizzle), fp32 rows 128 bytes (128-byte swizzle).
gemm_status_t encode_output(CUtensorMap *map, void *ptr, int64_t cols, int64_t rows, int64_t ld, bool bf16) {
    const int esize = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t elem_strides[2] = {1, 1};
    CUresult r = g_encode_tiled(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr,
                                dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

// Grow the workspace to at least `bytes`; the caller holds ds.ws_mutex.
gemm_status_t ensure_workspace(DeviceState &ds, size_t bytes) {
    if (ds.workspace_bytes >= bytes) return GEMM_OK;
    if (ds.workspace) {
        cudaDeviceSynchronize();   // the old buffer may still be read by queued work
        cudaFree(ds.workspace);
        ds.workspace = nullptr;
        ds.workspace_bytes = 0;
    }
    void *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_OUT_OF_MEMORY;
    }
    ds.workspace = static_cast<float *>(p);
    ds.workspace_bytes = bytes;
    return GEMM_OK;
}

gemm_status_t ensure_flags(DeviceState &ds) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ds.sk_flags) return GEMM_OK;
    void *p = nullptr;
    const size_t bytes = static_cast<size_t>(kMaxFlagSlots) * 4;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemset(p, 0, bytes) != cudaSuccess) {
        cudaFree(p);
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    ds.sk_flags = static_cast<unsigned int *>(p);
    return GEMM_OK;
}

unsigned int next_epoch(DeviceState &ds) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (++ds.epoch == 0) ds.epoch = 1;   // 0 is the value of fresh flags
    return ds.epoch;
}

// The fused epilogue an options struct asks for; epi = 0 when there is none
// or it is the identity (alpha 1, beta 0, no bias, no activation).
EpilogueArgs epilogue_args(const gemm_options_t &o) {
    EpilogueArgs e{0, 1.0f, 0.0f, nullptr, GEMM_ACT_NONE};
    if (!o.epilogue) return e;
    const gemm_epilogue_t &x = *o.epilogue;
    e.alpha = x.alpha;
    e.beta = x.beta;
    e.bias = x.bias;
    e.act = x.activation;
    e.epi = (x.alpha != 1.0f || x.beta != 0.0f || x.bias != nullptr || x.activation != GEMM_ACT_NONE) ? 1 : 0;
    return e;
}

gemm_status_t check_epilogue(const gemm_options_t &o) {
    if (!o.epilogue) return GEMM_OK;
    const gemm_epilogue_t &x = *o.epilogue;
    if (x.activation < GEMM_ACT_NONE || x.activation > GEMM_ACT_GELU) return GEMM_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(x.bias) % 16 != 0) return GEMM_ERR_MISALIGNED;
    return GEMM_OK;
}

// K == 0: C := 0, or with a fused epilogue C := act(beta * C + bias).
gemm_status_t launch_fill_zero(int64_t M, int64_t N, void *C, int64_t ldc, int esize, int num_sms,
                               cudaStream_t stream, const EpilogueArgs &ep) {
    const long long total = M * N;
    long long blocks = (total + 255) / 256;
    if (blocks > 4LL * num_sms) blocks = 4LL * num_sms;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaError_t e;
    if (ep.epi) {
        e = cudaLaunchKernelEx(&cfg, epilogue_only_kernel, C, static_cast<long long>(ldc), static_cast<int>(M),
                               static_cast<int>(N), esize == 2 ? 1 : 0, ep);
    } else {
        e = cudaLaunchKernelEx(&cfg, fill_zero_kernel, C, static_cast<long long>(ldc), static_cast<int>(M),
                               static_cast<int>(N), esize);
    }
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

// Checks shared by every GEMM entry point; no CUDA calls.  Leading
// dimensions: A row-major lda >= K, column-major lda >= M; B column-major
// ldb >= K, row-major ldb >= N.
gemm_status_t check_operands(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                             const void *C, int64_t ldc, gemm_layout_t layout_a, gemm_layout_t layout_b,
                             gemm_dtype_t out_dtype) {
    const int esize = out_dtype == GEMM_OUT_BF16 ? 2 : 4;
    if (!C || ldc < N) return GEMM_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(C) % 16 != 0 || (ldc * esize) % 16 != 0) return GEMM_ERR_MISALIGNED;
    if (K > 0) {
        const int64_t min_lda = layout_a == GEMM_ROW_MAJOR ? K : M;
        const int64_t min_ldb = layout_b == GEMM_COL_MAJOR ? K : N;
        if (!A || !B || lda < min_lda || ldb < min_ldb) return GEMM_ERR_INVALID_VALUE;
        if (reinterpret_cast<uintptr_t>(A) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0 || lda % 8 != 0 ||
            ldb % 8 != 0)
            return GEMM_ERR_MISALIGNED;
    }
    return GEMM_OK;
}

// Where the split-K partial sums of one call go.
struct PartialBuffer {
    bool fixed;          // true: the caller-provided array below, never grown
    float *ptr;
    int64_t floats;      // capacity when fixed
};

// Plan and enqueue one GEMM whose arguments have passed check_problem and
// check_operands, with M, N, K > 0.
// A convolution's implicit GEMM: the problem and the output extent.
struct ConvLaunch {
    const gemm_conv2d_desc_t *d;
    int64_t P, Q;
    int ncb;   // 64-channel blocks per tap
};

// x (N x H x W x C, NHWC) as an im2col tensor map: a load at window origin
// (c, w, h, n) with tap offsets (s dil_w, r dil_h) brings `rows` consecutive
// output pixels x 64 channels.  The pixel box runs over the window origins:
// from -pad to the last origin whose filter still fits the padded image
// (lower corner -pad, upper corner pad - dil (filter - 1)), stepping by the
// convolution's strides; pixels outside the image read as zero.
gemm_status_t encode_im2col(CUtensorMap *map, const void *x, const gemm_conv2d_desc_t &d, int rows) {
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d.C), static_cast<cuuint64_t>(d.W), static_cast<cuuint64_t>(d.H),
                          static_cast<cuuint64_t>(d.N)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d.C) * 2, static_cast<cuuint64_t>(d.W * d.C) * 2,
                             static_cast<cuuint64_t>(d.H * d.W * d.C) * 2};
    int lower[2] = {-d.pad_w, -d.pad_h};
    int upper[2] = {d.pad_w - d.dil_w * static_cast<int>(d.S - 1), d.pad_h - d.dil_h * static_cast<int>(d.R - 1)};
    cuuint32_t elem_strides[4] = {1, static_cast<cuuint32_t>(d.stride_w), static_cast<cuuint32_t>(d.stride_h), 1};
    CUresult r = g_encode_im2col(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(x), dims, strides, lower,
                                 upper, static_cast<cuuint32_t>(TILE_K), static_cast<cuuint32_t>(rows), elem_strides,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_VALUE;
}

// The filter (K x R x S x C, KRSC) as a 3-D tensor map (channels, taps,
// output channels), read in boxes of 64 channels x 1 tap x `box_rows` output
// channels: channels past C and output channels past K read as zero.
gemm_status_t encode_filter(CUtensorMap *map, const void *w, int64_t C, int64_t taps, int64_t K, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(taps), static_cast<cuuint64_t>(K)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2, static_cast<cuuint64_t>(taps * C) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(TILE_K), 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(w), dims, strides, box,
                                elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

gemm_status_t launch_gemm(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                          void *C, int64_t ldc, gemm_layout_t layout_a, gemm_layout_t layout_b,
                          gemm_dtype_t out_dtype, const gemm_options_t &o, cudaStream_t s, DeviceState &ds,
                          const PartialBuffer &pb, const ConvLaunch *conv = nullptr) {
    const int variant = choose_variant(M, N, K, o.kernel_variant, o.split_k, ds.desc);
    const VariantInfo vi = variant_info(variant);
    gemm_plan_t plan;
    gemm_status_t st = make_plan(M, N, K, layout_a, layout_b, out_dtype, o, !pb.fixed, ds.desc,
                                 kernel_desc(variant, ds.var[variant]), &plan);
    if (st != GEMM_OK) return st;
    const int64_t clusters = plan.launch_ctas / vi.cta_group;
    float *partials = nullptr;
    // held until the kernels that read the workspace are enqueued
    std::unique_lock<std::mutex> ws_lock(ds.ws_mutex, std::defer_lock);
    if (plan.stream_k_tiles > 0 || (plan.split_k > 1 && !pb.fixed)) ws_lock.lock();
    if (plan.stream_k_tiles > 0) {
        if (clusters * vi.cta_group * EPI_WARPS > kMaxFlagSlots) return GEMM_ERR_NOT_SUPPORTED;
        st = ensure_flags(ds);
        if (st != GEMM_OK) return st;
        st = ensure_workspace(ds, static_cast<size_t>(plan.workspace_bytes));
        if (st != GEMM_OK) return st;
    }
    if (plan.split_k > 1) {
        if (pb.fixed) {
            const int64_t per_split = plan.tiles * vi.tile_m * vi.bn;   // padded tiles; < 2^62
            if (per_split > pb.floats || plan.split_k > pb.floats / per_split) return GEMM_ERR_INVALID_VALUE;
            partials = pb.ptr;
        } else {
            st = ensure_workspace(ds, static_cast<size_t>(plan.workspace_bytes));
            if (st != GEMM_OK) return st;
            partials = ds.workspace;
        }
    }

    CUtensorMap tmap_a, tmap_b, tmap_c;
    const bool a_mn = layout_a == GEMM_COL_MAJOR, b_mn = layout_b == GEMM_ROW_MAJOR;
    if (conv) {
        const gemm_conv2d_desc_t &d = *conv->d;
        st = encode_im2col(&tmap_a, A, d, CTA_ROWS);
        if (st != GEMM_OK) return st;
        st = encode_filter(&tmap_b, B, d.C, d.R * d.S, d.K, vi.b_rows);
        if (st != GEMM_OK) return st;
    } else {
        st = a_mn ? encode_operand(&tmap_a, A, M, K, lda, vi.tile_k) : encode_operand(&tmap_a, A, K, M, lda, CTA_ROWS);
        if (st != GEMM_OK) return st;
        st = b_mn ? encode_operand(&tmap_b, B, N, K, ldb, vi.tile_k) : encode_operand(&tmap_b, B, K, N, ldb, vi.b_rows);
        if (st != GEMM_OK) return st;
    }
    st = encode_output(&tmap_c, C, N, M, ldc, out_dtype == GEMM_OUT_BF16);
    if (st != GEMM_OK) return st;
    // Stores by TMA stop at the last whole 16-byte piece of a row (the rest
    // of the row inside N is stored lane by lane); loads of the previous C
    // take the exact extent.
    const int64_t n_tma = N / (out_dtype == GEMM_OUT_BF16 ? 8 : 4) * (out_dtype == GEMM_OUT_BF16 ? 8 : 4);
    CUtensorMap tmap_out = tmap_c;
    if (n_tma > 0 && n_tma != N) {
        st = encode_output(&tmap_out, C, n_tma, M, ldc, out_dtype == GEMM_OUT_BF16);
        if (st != GEMM_OK) return st;
    }

    KernelParams p{};
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((M + vi.tile_m - 1) / vi.tile_m);
    p.tiles_n = static_cast<int>((N + vi.bn - 1) / vi.bn);
    p.k_tiles = plan.k_tiles;
    p.split_k = plan.split_k;
    p.group_m = plan.raster_group_m;
    p.num_units = plan.tiles * plan.split_k;
    p.out = C;
    p.ld_out = ldc;
    p.out_bf16 = out_dtype == GEMM_OUT_BF16 ? 1 : 0;
    p.n_tma = static_cast<int>(n_tma);
    p.partials = partials;
    if (o.timeout_ms > 0) {
        p.timeout_ns = static_cast<unsigned long long>(o.timeout_ms) * 1000000ull;
    } else {
        // k-tiles one wait may span: a work unit, plus a stream-K range
        const long long span = static_cast<long long>(plan.k_tiles_per_split) +
                               (plan.stream_k_tiles > 0 ? (plan.stream_k_tiles * plan.k_tiles + clusters - 1) / clusters : 0);
        p.timeout_ns = static_cast<unsigned long long>(DEFAULT_TIMEOUT_MS) * 1000000ull +
                       static_cast<unsigned long long>(span) * DEFAULT_TIMEOUT_US_PER_K_TILE * 1000ull;
    }
    p.skip_load = o.debug_skip_load;
    p.a_mn = a_mn ? 1 : 0;
    p.b_mn = b_mn ? 1 : 0;
    if (conv) {
        const gemm_conv2d_desc_t &d = *conv->d;
        p.conv = 1;
        p.cv_S = static_cast<int>(d.S);
        p.cv_PQ = static_cast<int>(conv->P * conv->Q);
        p.cv_Q = static_cast<int>(conv->Q);
        p.cv_taps = static_cast<int>(d.R * d.S);
        p.pad_h = d.pad_h;
        p.pad_w = d.pad_w;
        p.str_h = d.stride_h;
        p.str_w = d.stride_w;
        p.dil_h = d.dil_h;
        p.dil_w = d.dil_w;
        p.ncb = conv->ncb;
    }
    const EpilogueArgs ep = epilogue_args(o);
    p.epi = ep.epi;
    p.alpha = ep.alpha;
    p.beta = ep.beta;
    p.bias = ep.bias;
    p.act = ep.act;
    p.num_clusters = static_cast<int>(clusters);
    p.dp_tiles = static_cast<int>(plan.dp_tiles);
    p.sk_tiles = static_cast<int>(plan.stream_k_tiles);
    p.sk_iters = plan.stream_k_tiles * plan.k_tiles;
    if (plan.stream_k_tiles > 0) {
        if (clusters > SK_MAX_CLUSTERS) return GEMM_ERR_NOT_SUPPORTED;   // the plan never asks for this
        int64_t bounds[SK_MAX_CLUSTERS + 1];
        stream_k_bounds(p.sk_iters, clusters, plan.k_tiles, o, bounds);
        for (int64_t c = 0; c <= clusters; ++c) p.sk_bounds[c] = bounds[c];
        p.partials = ds.workspace;
        p.sk_flags = ds.sk_flags;
        p.epoch = next_epoch(ds);
    }

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.launch_ctas));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = vi.smem;
    cfg.stream = s;
    // Programmatic stream serialisation: this launch may begin while the
    // previous kernel in the stream finishes (see grid_dependency_wait).
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1] = cluster_attr(vi.cta_group);
    cfg.attrs = attrs;
    cfg.numAttrs = vi.cta_group > 1 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kernel_fn(variant), tmap_a, tmap_b, tmap_c, tmap_out, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (o.mainloop_done_event && cudaEventRecord(static_cast<cudaEvent_t>(o.mainloop_done_event), s) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    if (plan.split_k > 1) {
        const long long total = plan.tiles * vi.tile_m * vi.bn / 4;   // float4s per slice
        long long blocks = (total + 31) / 32;
        const long long cap = 8LL * ds.desc.num_sms;
        if (blocks > cap) blocks = cap;
        cudaLaunchConfig_t cc{};
        cc.gridDim = dim3(static_cast<unsigned>(blocks));
        cc.blockDim = dim3(COMBINE_WARPS * 32);
        cc.stream = s;
        cudaLaunchAttribute pdl{};
        pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl.val.programmaticStreamSerializationAllowed = 1;
        cc.attrs = &pdl;
        cc.numAttrs = 1;
        const int per_warp = (plan.split_k + COMBINE_WARPS - 1) / COMBINE_WARPS;
        auto combine = per_warp <= 2 ? splitk_combine_kernel<2>
                     : per_warp <= 4 ? splitk_combine_kernel<4>
                     : per_warp <= 8 ? splitk_combine_kernel<8>
                     : per_warp <= 16 ? splitk_combine_kernel<16> : splitk_combine_kernel<24>;
        if (cudaLaunchKernelEx(&cc, combine, static_cast<const float *>(partials), plan.split_k,
                               static_cast<long long>(plan.tiles), p.tiles_n, vi.tile_m, vi.bn, static_cast<int>(M),
                               static_cast<int>(N), C, static_cast<long long>(ldc),
                               out_dtype == GEMM_OUT_BF16 ? 1 : 0, ep) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    }
    return GEMM_OK;
}

gemm_status_t current_device(int *device, DeviceState **ds) {
    if (cudaGetDevice(device) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    return device_state(*device, ds);
}

}  // namespace

}  // namespace gemm

using namespace gemm;

extern "C" {

gemm_status_t gemm_device_desc_query(int device, gemm_device_desc_t *dev) {
    if (!dev) return GEMM_ERR_INVALID_VALUE;
    std::memset(dev, 0, sizeof *dev);
    return query_desc(device, dev);
}

gemm_status_t gemm_kernel_desc(int kernel_variant, gemm_kernel_desc_t *kern) {
    if (!kern || kernel_variant < 0 || kernel_variant >= VARIANT_COUNT) return GEMM_ERR_INVALID_VALUE;
    const int v = resolve_variant(kernel_variant);
    VariantState vs;
    int device = 0;
    DeviceState *ds = nullptr;
    if (current_device(&device, &ds) == GEMM_OK) vs = ds->var[v];
    cudaGetLastError();
    *kern = kernel_desc(v, vs);
    return GEMM_OK;
}

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, gemm_layout_t layout_a, gemm_layout_t layout_b,
                        gemm_dtype_t out_dtype, const gemm_options_t *opts, gemm_plan_t *plan) {
    if (!plan) return GEMM_ERR_INVALID_VALUE;
    gemm_options_t o{};
    if (opts) o = *opts;
    gemm_status_t st = check_problem(M, N, K, layout_a, layout_b, out_dtype, o.split_k);
    if (st != GEMM_OK) return st;
    if (o.kernel_variant < 0 || o.kernel_variant >= VARIANT_COUNT) return GEMM_ERR_INVALID_VALUE;
    int device = 0;
    DeviceState *ds = nullptr;
    st = current_device(&device, &ds);
    if (st != GEMM_OK) return st;
    const int v = choose_variant(M, N, K, o.kernel_variant, o.split_k, ds->desc);
    return make_plan(M, N, K, layout_a, layout_b, out_dtype, o, true, ds->desc, kernel_desc(v, ds->var[v]), plan);
}

gemm_status_t gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                           void *C, int64_t ldc, gemm_layout_t layout_a, gemm_layout_t layout_b,
                           gemm_dtype_t out_dtype, const gemm_options_t *opts, void *stream) {
    gemm_options_t o{};
    if (opts) o = *opts;
    gemm_status_t st = check_problem(M, N, K, layout_a, layout_b, out_dtype, o.split_k);
    if (st != GEMM_OK) return st;
    if (o.timeout_ms < 0 || o.raster_group_m < 0 || o.debug_skip_load < 0 || o.kernel_variant < 0 ||
        o.kernel_variant >= VARIANT_COUNT)
        return GEMM_ERR_INVALID_VALUE;
    st = check_epilogue(o);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    st = check_operands(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype);
    if (st != GEMM_OK) return st;

    int device = 0;
    DeviceState *ds = nullptr;
    st = current_device(&device, &ds);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return launch_fill_zero(M, N, C, ldc, out_dtype == GEMM_OUT_BF16 ? 2 : 4, ds->desc.num_sms, s, epilogue_args(o));
    return launch_gemm(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype, o, s, *ds,
                       PartialBuffer{false, nullptr, 0});
}

gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                        void *C, int64_t ldc, gemm_layout_t layout_a, gemm_layout_t layout_b, gemm_dtype_t out_dtype,
                        int split_k, void *stream) {
    gemm_options_t o{};
    o.split_k = split_k;
    return gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype, &o, stream);
}

gemm_status_t gemm_reserve_workspace(size_t bytes) {
    int device = 0;
    DeviceState *ds = nullptr;
    gemm_status_t st = current_device(&device, &ds);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lock(ds->ws_mutex);
    return ensure_workspace(*ds, bytes);
}

void gemm_release_workspace(void) {
    release_host_staging();   // takes its own per-device locks, never under a workspace lock
    int current = -1;
    if (cudaGetDevice(&current) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    for (int d = 0; d < kMaxDevices; ++d) {
        DeviceState &ds = g_devices[d];
        std::lock_guard<std::mutex> lock(ds.ws_mutex);
        if (!ds.workspace) continue;
        if (cudaSetDevice(d) == cudaSuccess) {
            cudaDeviceSynchronize();
            cudaFree(ds.workspace);
        }
        ds.workspace = nullptr;
        ds.workspace_bytes = 0;
    }
    cudaSetDevice(current);
}

gemm_status_t gemm_get_device_status(void *stream, unsigned int *where) {
    if (where) *where = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    unsigned int w = 0;
    if (cudaMemcpyFromSymbol(&w, g_fault_word, sizeof w) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (w != 0) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_fault_word, &zero, sizeof zero);
    }
    if (where) *where = w;
    return w != 0 ? GEMM_ERR_DEVICE_TIMEOUT : GEMM_OK;
}

}  // extern "C"

// ------------------------------------------------ convolution (implicit GEMM)

namespace gemm {
namespace {

// The implicit GEMM of a convolution: M = N P Q, N = K, K = R S (C rounded up
// to 64-channel blocks); the options as given.
struct ConvProblem {
    ConvLaunch launch;
    int64_t M, N, K;
    gemm_options_t o;
};

gemm_status_t conv_problem(const gemm_conv2d_desc_t *d, const gemm_options_t *opts, ConvProblem *cp) {
    int64_t P = 0, Q = 0;
    gemm_status_t st = conv_check(d, &P, &Q);
    if (st != GEMM_OK) return st;
    gemm_options_t o{};
    if (opts) o = *opts;
    if (o.kernel_variant < 0 || o.kernel_variant >= VARIANT_COUNT) return GEMM_ERR_INVALID_VALUE;
    // the im2col pixel box of a 4-D tensor map spans corners in [-128, 127]
    if (d->pad_h > 127 || d->pad_w > 127 || d->dil_h * (d->R - 1) > 127 || d->dil_w * (d->S - 1) > 127)
        return GEMM_ERR_NOT_SUPPORTED;
    const int ncb = static_cast<int>((d->C + TILE_K - 1) / TILE_K);
    cp->launch = ConvLaunch{d, P, Q, ncb};
    cp->M = d->N * P * Q;
    cp->N = d->K;
    cp->K = d->R * d->S * ncb * TILE_K;
    cp->o = o;
    return GEMM_OK;
}

}  // namespace
}  // namespace gemm

extern "C" gemm_status_t gemm_conv2d_plan(const gemm_conv2d_desc_t *d, gemm_dtype_t out_dtype,
                                          const gemm_options_t *opts, gemm_plan_t *plan) {
    if (!plan) return GEMM_ERR_INVALID_VALUE;
    ConvProblem cp;
    gemm_status_t st = conv_problem(d, opts, &cp);
    if (st != GEMM_OK) return st;
    st = check_problem(cp.M, cp.N, cp.K, GEMM_ROW_MAJOR, GEMM_COL_MAJOR, out_dtype, cp.o.split_k);
    if (st != GEMM_OK) return st;
    int device = 0;
    DeviceState *ds = nullptr;
    st = current_device(&device, &ds);
    if (st != GEMM_OK) return st;
    const int v = choose_variant(cp.M, cp.N, cp.K, cp.o.kernel_variant, cp.o.split_k, ds->desc);
    return make_plan(cp.M, cp.N, cp.K, GEMM_ROW_MAJOR, GEMM_COL_MAJOR, out_dtype, cp.o, true, ds->desc,
                     kernel_desc(v, ds->var[v]), plan);
}

extern "C" gemm_status_t gemm_conv2d_fprop_bf16(const gemm_conv2d_desc_t *d, const void *x, const void *w, void *y,
                                                gemm_dtype_t out_dtype, const gemm_options_t *opts, void *stream) {
    ConvProblem cp;
    gemm_status_t st = conv_problem(d, opts, &cp);
    if (st != GEMM_OK) return st;
    const gemm_options_t &o = cp.o;
    st = check_problem(cp.M, cp.N, cp.K, GEMM_ROW_MAJOR, GEMM_COL_MAJOR, out_dtype, o.split_k);
    if (st != GEMM_OK) return st;
    if (o.timeout_ms < 0 || o.raster_group_m < 0 || o.debug_skip_load != 0) return GEMM_ERR_INVALID_VALUE;
    st = check_epilogue(o);
    if (st != GEMM_OK) return st;
    if (!x || !w || !y) return GEMM_ERR_INVALID_VALUE;
    const int esize = out_dtype == GEMM_OUT_BF16 ? 2 : 4;
    if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(w) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(y) % 16 != 0 || d->C % 8 != 0 || (d->K * esize) % 16 != 0)
        return GEMM_ERR_MISALIGNED;

    int device = 0;
    DeviceState *ds = nullptr;
    st = current_device(&device, &ds);
    if (st != GEMM_OK) return st;
    return launch_gemm(cp.M, cp.N, cp.K, x, d->C, w, cp.K, y, d->K, GEMM_ROW_MAJOR, GEMM_COL_MAJOR, out_dtype, o,
                       static_cast<cudaStream_t>(stream), *ds, PartialBuffer{false, nullptr, 0}, &cp.launch);
}

// ------------------------------------------- split-K without device allocation
//
// gemm_bf16_splitk_noalloc (contract in gemm_bf16.h): the same kernels as
// gemm_bf16, with the split-K partial sums in a fixed array compiled into the
// library instead of the cudaMalloc'd workspace.

namespace gemm {

// Host code must not use this name as a device address: on the host it is only
// a stand-in.  The device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) float g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_FLOATS];

namespace {

std::mutex g_noalloc_mutex;
float *g_noalloc_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current),
// looked up once per device.
gemm_status_t noalloc_scratch(int device, float **out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_scratch_addr[device]) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        g_noalloc_scratch_addr[device] = static_cast<float *>(addr);
    }
    *out = g_noalloc_scratch_addr[device];
    return GEMM_OK;
}

}  // namespace
}  // namespace gemm

extern "C" gemm_status_t gemm_bf16_splitk_noalloc(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                                                  const void *B, int64_t ldb, void *C, int64_t ldc,
                                                  gemm_layout_t layout_a, gemm_layout_t layout_b,
                                                  gemm_dtype_t out_dtype, int split_k, void *stream) {
    gemm_status_t st = check_problem(M, N, K, layout_a, layout_b, out_dtype, split_k);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    st = check_operands(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype);
    if (st != GEMM_OK) return st;

    int device = 0;
    DeviceState *ds = nullptr;
    st = current_device(&device, &ds);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return launch_fill_zero(M, N, C, ldc, out_dtype == GEMM_OUT_BF16 ? 2 : 4, ds->desc.num_sms, s, EpilogueArgs{0, 1.0f, 0.0f, nullptr, GEMM_ACT_NONE});

    float *scratch = nullptr;
    st = noalloc_scratch(device, &scratch);
    if (st != GEMM_OK) return st;
    gemm_options_t o{};
    o.split_k = split_k;
    return launch_gemm(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype, o, s, *ds,
                       PartialBuffer{true, scratch, static_cast<int64_t>(GEMM_NOALLOC_SCRATCH_FLOATS)});
}
