// Host-side planning: argument checks, the closed forms of the launch and
// the occupancy arithmetic.  No CUDA calls; see gemm_bf16.h for the contract.
//
// Closed forms: chapter 10 "Tensor Cores, shapes, and tile alignment",
// sections "Shape the operation" (FLOPs = 2MNK, G = ceil(M/T_M) ceil(N/T_N),
// eta_wave = G / (ceil(G/(S b)) S b)), "Padding efficiency"
// (eta_pad = MNK / (M'N'K')) and "When shape alone can't fix wave
// efficiency" (split-K multiplies the CTAs).  Occupancy: "Grid 24 is not
// headroom", section "The question I never asked" (registers per CTA =
// per-thread count, granted in multiples of 8, times the threads; b is the
// tightest of registers and shared memory).
#include "gemm_bf16.h"
#include "plan_internal.h"
#include "kernel_config.h"

#include <climits>
#include <cstring>

namespace gemm {

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

gemm_status_t check_problem(int64_t M, int64_t N, int64_t K, gemm_layout_t la, gemm_layout_t lb,
                            gemm_dtype_t out, int split_k) {
    if (M < 0 || N < 0 || K < 0 || M > INT_MAX || N > INT_MAX || K > INT_MAX) return GEMM_ERR_INVALID_VALUE;
    if ((la != GEMM_ROW_MAJOR && la != GEMM_COL_MAJOR) || (lb != GEMM_ROW_MAJOR && lb != GEMM_COL_MAJOR))
        return GEMM_ERR_INVALID_VALUE;
    if (out != GEMM_OUT_F32 && out != GEMM_OUT_BF16) return GEMM_ERR_INVALID_VALUE;
    if (split_k < 0) return GEMM_ERR_INVALID_VALUE;
    return GEMM_OK;
}

// A convolution's fields and output extent (see gemm_conv2d_desc_t).
gemm_status_t conv_check(const gemm_conv2d_desc_t *d, int64_t *P, int64_t *Q) {
    if (!d) return GEMM_ERR_INVALID_VALUE;
    const int64_t big = INT_MAX;
    if (d->N < 1 || d->H < 1 || d->W < 1 || d->C < 1 || d->K < 1 || d->R < 1 || d->S < 1) return GEMM_ERR_INVALID_VALUE;
    if (d->N > big || d->H > big || d->W > big || d->C > big || d->K > big || d->R > big || d->S > big)
        return GEMM_ERR_INVALID_VALUE;
    if (d->pad_h < 0 || d->pad_w < 0 || d->stride_h < 1 || d->stride_w < 1 || d->dil_h < 1 || d->dil_w < 1)
        return GEMM_ERR_INVALID_VALUE;
    const int64_t p = (d->H + 2 * static_cast<int64_t>(d->pad_h) - d->dil_h * (d->R - 1) - 1);
    const int64_t q = (d->W + 2 * static_cast<int64_t>(d->pad_w) - d->dil_w * (d->S - 1) - 1);
    if (p < 0 || q < 0) return GEMM_ERR_INVALID_VALUE;   // the filter does not fit the padded image
    const int64_t Pv = p / d->stride_h + 1, Qv = q / d->stride_w + 1;
    // N P Q, the padded R S C and the input's element count stay in int range
    if (d->N * Pv > big || d->N * Pv * Qv > big || d->R * d->S > big || d->R * d->S * cdiv(d->C, TILE_K) * TILE_K > big ||
        d->N * d->H > big || d->N * d->H * d->W > big)
        return GEMM_ERR_INVALID_VALUE;
    if (P) *P = Pv;
    if (Q) *Q = Qv;
    return GEMM_OK;
}

int round_regs(int regs_per_thread) { return (regs_per_thread + 7) / 8 * 8; }

gemm_status_t occupancy(const gemm_kernel_desc_t &k, const gemm_device_desc_t &d, int *b_out, int *lim_out) {
    *b_out = 0;
    *lim_out = GEMM_LIMIT_BLOCKS;
    if (k.threads_per_cta <= 0 || k.smem_per_cta < 0 || k.tmem_cols_per_cta < 0 || k.regs_per_thread < 0)
        return GEMM_ERR_INVALID_VALUE;
    const int64_t big = INT_MAX;
    int64_t by_regs = big, by_smem = big, by_tmem = big;
    if (k.regs_per_thread > 0) by_regs = d.regs_per_sm / ((int64_t)round_regs(k.regs_per_thread) * k.threads_per_cta);
    const int64_t smem_cost = (int64_t)k.smem_per_cta + d.smem_reserved_per_cta;
    if (smem_cost > 0) by_smem = d.smem_per_sm / smem_cost;
    if (k.tmem_cols_per_cta > 0) by_tmem = d.tmem_cols_per_sm / k.tmem_cols_per_cta;
    int64_t by_threads = d.max_threads_per_sm / k.threads_per_cta;
    int64_t by_blocks = d.max_ctas_per_sm;
    const int64_t vals[5] = {by_regs, by_smem, by_tmem, by_threads, by_blocks};
    const int names[5] = {GEMM_LIMIT_REGISTERS, GEMM_LIMIT_SMEM, GEMM_LIMIT_TMEM, GEMM_LIMIT_THREADS,
                          GEMM_LIMIT_BLOCKS};
    int64_t b = vals[0];
    for (int i = 1; i < 5; ++i) b = b < vals[i] ? b : vals[i];
    for (int i = 0; i < 5; ++i) {
        if (vals[i] == b) { *lim_out = names[i]; break; }
    }
    if (k.smem_per_cta > d.smem_optin_per_cta) b = 0;
    *b_out = (int)b;
    return b > 0 ? GEMM_OK : GEMM_ERR_INVALID_VALUE;
}

int choose_split(int64_t tiles, int k_tiles, int capacity, int requested, int64_t K) {
    if (k_tiles <= 0) return 1;
    int s;
    if (requested > 0) {
        s = requested;
    } else {
        // Automatic: only for few tiles and a long enough K (see
        // AUTO_SPLIT_MIN_K); then give each slot a slice of K, keeping slices
        // at least MIN_K_TILES_PER_SPLIT k-tiles long.
        s = 1;
        if ((tiles * 8 <= capacity && K >= AUTO_SPLIT_MIN_K) || (tiles * 4 <= capacity && K >= LONG_K)) {
            int64_t by_slots = capacity / tiles;
            int64_t by_k = k_tiles / MIN_K_TILES_PER_SPLIT;
            int64_t c = by_slots < by_k ? by_slots : by_k;
            s = c > 1 ? (int)c : 1;
        }
    }
    if (s > k_tiles) s = k_tiles;
    return s < 1 ? 1 : s;
}

int resolve_variant(int requested) {
    if (requested == VARIANT_AUTO) return VARIANT_2SM_256x256;
    return requested;
}

// The automatic choice between the single-CTA 128x256 and the pair 256x256
// kernels: both spend the same time on 64 of K of one tile, so compare the
// 64-wide k-steps each resident cluster would run with the work spread evenly,
// ceil(T * k_tiles / C) -- T tiles, C = S single CTAs or S/2 pairs -- and
// give the pair kernel the advantage it shows at equal work (its tensor
// pipes stay about 7 % busier: half the B traffic per SM, a deeper ring).
int choose_variant(int64_t M, int64_t N, int64_t K, int requested, int split_k, const gemm_device_desc_t &dev) {
    if (requested != VARIANT_AUTO) return requested;
    const int64_t kb = cdiv(K, TILE_K) > 0 ? cdiv(K, TILE_K) : 1;
    const int64_t c1 = dev.num_sms > 0 ? dev.num_sms : 1;
    const int64_t c2 = dev.num_sms / 2 > 0 ? dev.num_sms / 2 : 1;
    // A small GEMM (256 x 128 pair tiles filling at most half the pairs, a K
    // too short for the plan to split) is latency-bound: the smaller pair
    // tiles spread it over more SMs and shorten each CTA's epilogue
    // (measured: 512^3 7.8 against 9.2 us, 1024^3 10.4 against 11.4 us).
    if (split_k <= 1 && K < AUTO_SPLIT_MIN_K && cdiv(M, 256) * cdiv(N, 128) * 2 <= c2) return VARIANT_2SM_256x128;
    // One tile row (M <= 128) with a long K: 128 x 128 tiles give twice the
    // work units of 128 x 256 tiles, so a split that fills the SMs takes half
    // the slices, each CTA stores half a partial tile and the combine reads
    // half as much -- but each tile of the row reads A again.  The two plans
    // (each with its own split: the one asked for, or the plan's own) are
    // compared by an estimate of their time: the operand bytes one CTA
    // streams at about 100 GB/s per SM, at least the unique operand bytes at
    // about 6.8 TB/s, plus, when K is split, about 6 us (the combine kernel,
    // a kernel boundary) and the fp32 partial tiles written and read back at
    // about 2 TB/s.  Within 0.5 us the plan with more work units wins.  The
    // 128 x 128 plan must fit in one wave.  (Measured, us, 128 x 128 against
    // 128 x 256 or the pair kernel: 128 x 256 x 65536 with the plan's split
    // 15.9 against 16.4, split 74 15.9 against 19.2, split 1 324 against 385;
    // 128 x 1024 x 4096 11.3 against 12.4; 100 x 3000 x 2048 15.1 against
    // 16.6; the other way, where the 128 x 128 plan cannot split:
    // 64 x 4096 x 4096 24.8 against 19.9, 128 x 8192 x 8192 46.7 against
    // 46.0.)
    if (M <= 128 && N > 128 && K >= AUTO_SPLIT_MIN_K) {
        const int64_t t4 = cdiv(N, 128), t1 = cdiv(N, 256);
        auto split_for = [&](int64_t tiles) -> int64_t {
            return split_k > 0 ? (split_k < kb ? split_k : kb)
                               : choose_split(tiles, static_cast<int>(kb), static_cast<int>(c1), 0, K);
        };
        const int64_t s4 = split_for(t4), s1 = split_for(t1);
        const double unique_us = 2.0 * static_cast<double>(M * K + N * K) / 6.8e6;
        auto estimate_us = [&](int64_t bn, int64_t tiles, int64_t s) {
            const int64_t units = tiles * s;
            const int64_t waves = cdiv(units, c1);
            const double cta_bytes = (128.0 + static_cast<double>(bn)) * 2.0 * TILE_K *
                                     static_cast<double>(cdiv(kb, s) * waves);
            const double stream_us = cta_bytes / 1.0e5;
            const double split_us = s > 1 ? 6.0 + static_cast<double>(units) * 128.0 * bn * 4.0 / 2.0e6 : 0.0;
            return (stream_us > unique_us ? stream_us : unique_us) + split_us;
        };
        const double e4 = estimate_us(128, t4, s4), e1 = estimate_us(256, t1, s1);
        const bool tie = e4 - e1 < 0.5 && e1 - e4 < 0.5;
        if (t4 * s4 <= c1 && (tie ? t4 * s4 >= t1 * s1 : e4 < e1)) return VARIANT_1SM_128x128;
    }
    const int64_t t1 = cdiv(M, 128) * cdiv(N, 256), t2 = cdiv(M, 256) * cdiv(N, 256);
    int64_t w1, w2;
    if (split_k > 1) {   // a given split: rounds of work units times k-tiles per unit
        const int64_t s = split_k < kb ? split_k : kb;
        w1 = cdiv(t1 * s, c1) * cdiv(kb, s);
        w2 = cdiv(t2 * s, c2) * cdiv(kb, s);
    } else {
        w1 = cdiv(t1 * kb, c1);
        w2 = cdiv(t2 * kb, c2);
    }
    return w1 * 100 < w2 * 93 ? VARIANT_1SM_128x256 : VARIANT_2SM_256x256;
}

gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, gemm_layout_t la, gemm_layout_t lb,
                        gemm_dtype_t out, const gemm_options_t &o, bool allow_stream_k,
                        const gemm_device_desc_t &dev, const gemm_kernel_desc_t &kern, gemm_plan_t *plan) {
    gemm_status_t st = check_problem(M, N, K, la, lb, out, o.split_k);
    if (st != GEMM_OK) return st;
    if (o.kernel_variant < 0 || o.kernel_variant >= VARIANT_COUNT) return GEMM_ERR_INVALID_VALUE;
    if (dev.num_sms <= 0) return GEMM_ERR_INVALID_VALUE;
    const int v = choose_variant(M, N, K, o.kernel_variant, o.split_k, dev);
    const VariantInfo vi = variant_info(v);
    const int cs = kern.cluster_size > 0 ? kern.cluster_size : 1;
    if (cs != vi.cta_group) return GEMM_ERR_INVALID_VALUE;
    const bool persistent = o.non_persistent == 0;
    std::memset(plan, 0, sizeof *plan);
    int b = 0, lim = 0;
    st = occupancy(kern, dev, &b, &lim);
    if (st != GEMM_OK) return st;

    // CTAs resident at once: S b, rounded down to whole clusters, or the
    // device's own count of resident clusters when it is known.
    int64_t clusters = (int64_t)dev.num_sms * b / cs;
    if (kern.max_active_clusters > 0 && kern.max_active_clusters < clusters) clusters = kern.max_active_clusters;
    if (clusters <= 0) return GEMM_ERR_INVALID_VALUE;
    const int64_t resident = clusters * cs;

    plan->kernel_variant = v;
    plan->cluster_size = cs;
    plan->resident_ctas = resident;
    plan->tile_m = vi.tile_m;
    plan->tile_n = vi.bn;
    plan->tile_k = vi.tile_k;
    plan->stages = vi.stages;
    plan->threads_per_cta = kern.threads_per_cta;
    plan->num_sms = dev.num_sms;
    plan->ctas_per_sm = b;
    plan->occupancy_limiter = lim;
    plan->persistent = persistent ? 1 : 0;
    const int64_t T = cdiv(M, vi.tile_m) * cdiv(N, vi.bn);
    plan->tiles = T;
    plan->k_tiles = (int)cdiv(K, vi.tile_k);

    // Stream-K tail: only with the plan's own choice of split, on a persistent
    // grid (every cluster resident, as the hand-off between clusters needs),
    // when the tiles do not divide the clusters evenly -- and then when it
    // pays: at least one full wave, and a last wave whose idle share, in
    // 128-wide k-tiles of a 128 x 256 block per SM, reaches
    // STREAM_K_MIN_WASTE -- or always when asked (no_stream_k < 0).
    int64_t sk_tiles = 0;
    if (allow_stream_k && persistent && o.split_k == 0 && o.no_stream_k <= 0 && plan->k_tiles >= 2 && T > 0 &&
        T % clusters != 0 && clusters <= SK_MAX_CLUSTERS) {
        const double idle_k_tiles =
            (double)(cdiv(T, clusters) * clusters - T) / (double)clusters * plan->k_tiles;
        const double waste = idle_k_tiles * (vi.tile_k / 128.0) * ((double)vi.tile_m * vi.bn / cs / (128.0 * 256.0));
        const bool pays = T >= clusters && waste >= STREAM_K_MIN_WASTE;
        if (o.no_stream_k < 0 || pays) sk_tiles = T >= 2 * clusters ? clusters + T % clusters : T;
    }
    plan->stream_k_tiles = sk_tiles;
    plan->dp_tiles = T - sk_tiles;
    plan->split_k = (T > 0 && sk_tiles == 0) ? choose_split(T, plan->k_tiles, (int)clusters, o.split_k, K) : 1;
    plan->k_tiles_per_split = plan->k_tiles > 0 ? (int)cdiv(plan->k_tiles, plan->split_k) : 0;
    plan->grid = T * plan->split_k * cs;
    plan->launch_ctas = persistent ? (plan->grid < resident ? plan->grid : resident) : plan->grid;
    if (sk_tiles > 0) plan->launch_ctas = resident;   // every cluster takes a share of the tail
    plan->m_padded = cdiv(M, vi.tile_m) * vi.tile_m;
    plan->n_padded = cdiv(N, vi.bn) * vi.bn;
    plan->k_padded = cdiv(K, vi.tile_k) * vi.tile_k;
    if (plan->grid > 0) {
        const int64_t waves = cdiv(plan->grid, resident);
        plan->eta_wave = (double)plan->grid / ((double)waves * (double)resident);
    }
    if (sk_tiles > 0) {
        // the most k-iterations any cluster runs: its whole tiles (dealt round
        // robin) and its stream-K range
        int64_t bounds[SK_MAX_CLUSTERS + 1];
        stream_k_bounds(sk_tiles * plan->k_tiles, clusters, plan->k_tiles, o, bounds);
        int64_t worst = 0;
        for (int64_t c = 0; c < clusters; ++c) {
            const int64_t whole = plan->dp_tiles / clusters + (c < plan->dp_tiles % clusters ? 1 : 0);
            const int64_t its = whole * plan->k_tiles + bounds[c + 1] - bounds[c];
            if (its > worst) worst = its;
        }
        const double ideal = (double)T * plan->k_tiles / (double)clusters;
        plan->eta_stream_k = ideal / (double)worst;
    }
    if (M > 0 && N > 0 && K > 0) {
        plan->eta_pad = ((double)M / plan->m_padded) * ((double)N / plan->n_padded) * ((double)K / plan->k_padded);
    }
    plan->flops = 2.0 * (double)M * (double)N * (double)K;
    // Raster groups of 16 m-tiles; with at least eight waves of tiles, groups
    // of 8: the 76 tiles in flight then span about 8 m-tiles and 10 n-tiles
    // instead of 16 and 5, fewer operand bytes per wave (at 16384 x 8192 x
    // 8192, 2.14 against 2.50 GB read from DRAM, about 1 % faster).
    plan->raster_group_m = o.raster_group_m > 0 ? o.raster_group_m
                         : (persistent && T >= (int64_t)MANY_WAVES * clusters) ? MANY_WAVES_RASTER_GROUP_M
                                                                              : DEFAULT_RASTER_GROUP_M;
    plan->smem_bytes = vi.smem;
    plan->tmem_cols = vi.tmem_cols;
    if (plan->split_k > 1) {
        plan->workspace_bytes = (int64_t)plan->split_k * T * vi.tile_m * vi.bn * 4;
    } else if (sk_tiles > 0) {
        plan->workspace_bytes = clusters * (int64_t)vi.tile_m * vi.bn * 4;
    }
    return GEMM_OK;
}

// The sk_iters iterations are dealt out in contiguous ranges, the first
// (sk_iters mod clusters) ranges one longer.  A long epilogue -- GELU, or any
// that reads the previous C -- changes this:
//   - with k_tiles even (and at least 8) the ranges are made of whole half
//     tiles.  Every range then starts at k = 0 or k_tiles / 2 of a tile, so
//     clusters reading the same operand panels start on the same slices and
//     share them in L2, and no cluster runs a whole epilogue for a piece
//     shorter than half a tile.  The longest range may grow (4096^3: 48
//     iterations against 44; M = 4097: 64 against 51), and still: 4096^3
//     GELU(A.B + C + bias) 89.2 -> 87.2 us and A.B + C + bias 85.6 -> 83.6
//     against the tile-edge moves below; M = 4097 GELU 95.8 -> 94.6; the 3 x 3
//     convolutions with bias and GELU 76.7 -> 76.3 (28 x 28) and 80.0 -> 79.8
//     (56 x 56).  For the plain GEMM half tiles do not pay (4096^3 -0.7 %,
//     K = 4088 +0.6 %, M = 4097 +2.8 %, 28 x 28 convolution +5.5 %);
//   - otherwise a boundary within k_tiles / 4 of a tile's edge moves to the
//     edge, so that no cluster owns a tile for a few k-tiles of MMAs and still
//     runs its whole epilogue, nor starts with a sliver (4096^3 with even
//     ranges before: GELU(A.B + C + bias) 91.2 -> 87.5 us, A.B + C + bias
//     85.6 -> 84.4; for bias and ReLU alone 80.9 -> 81.2 and for the plain
//     GEMM 77.7 -> 79.3, so those keep even ranges).  A moved boundary never
//     passes a neighbour, as the move is less than half a tile.
void stream_k_bounds(int64_t sk_iters, int64_t clusters, int64_t k_tiles, const gemm_options_t &o, int64_t *bounds) {
    const bool long_epilogue =
        o.epilogue != nullptr && (o.epilogue->activation == GEMM_ACT_GELU || o.epilogue->beta != 0.0f);
    // contiguous ranges of whole units (sk_iters is a multiple of the unit), as even as they go
    const int64_t unit = long_epilogue && k_tiles >= 8 && k_tiles % 2 == 0 ? k_tiles / 2 : 1;
    const int64_t n = sk_iters / unit, base = n / clusters, rem = n % clusters;
    for (int64_t c = 0; c <= clusters; ++c) bounds[c] = unit * (c * base + (c < rem ? c : rem));
    const int64_t reach = k_tiles / 4;
    if (!long_epilogue || unit > 1 || reach == 0) return;
    for (int64_t c = 1; c < clusters; ++c) {
        const int64_t x = bounds[c], lo = x / k_tiles * k_tiles;
        if (x - lo <= reach) {
            bounds[c] = lo;
        } else if (lo + k_tiles - x <= reach && lo + k_tiles <= sk_iters) {
            bounds[c] = lo + k_tiles;
        }
    }
}

}  // namespace gemm

extern "C" {

gemm_status_t gemm_occupancy(const gemm_kernel_desc_t *kern, const gemm_device_desc_t *dev, int *ctas_per_sm,
                             int *limiter) {
    if (!kern || !dev || !ctas_per_sm || !limiter) return GEMM_ERR_INVALID_VALUE;
    return gemm::occupancy(*kern, *dev, ctas_per_sm, limiter);
}

gemm_status_t gemm_plan_for_device(int64_t M, int64_t N, int64_t K, gemm_layout_t layout_a, gemm_layout_t layout_b,
                                   gemm_dtype_t out_dtype, const gemm_options_t *opts, const gemm_device_desc_t *dev,
                                   const gemm_kernel_desc_t *kern, gemm_plan_t *plan) {
    if (!dev || !kern || !plan) return GEMM_ERR_INVALID_VALUE;
    gemm_options_t o{};
    if (opts) o = *opts;
    return gemm::make_plan(M, N, K, layout_a, layout_b, out_dtype, o, true, *dev, *kern, plan);
}

gemm_status_t gemm_conv2d_out_dims(const gemm_conv2d_desc_t *d, int64_t *P, int64_t *Q) {
    return gemm::conv_check(d, P, Q);
}

const char *gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE";
        case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
        case GEMM_ERR_NOT_SUPPORTED: return "GEMM_ERR_NOT_SUPPORTED";
        case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE";
        case GEMM_ERR_OUT_OF_MEMORY: return "GEMM_ERR_OUT_OF_MEMORY";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH";
        case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT";
    }
    return "GEMM_ERR_UNKNOWN";
}

const char *gemm_limiter_string(int limiter) {
    switch (limiter) {
        case GEMM_LIMIT_REGISTERS: return "registers";
        case GEMM_LIMIT_SMEM: return "smem";
        case GEMM_LIMIT_TMEM: return "tmem";
        case GEMM_LIMIT_THREADS: return "threads";
        case GEMM_LIMIT_BLOCKS: return "blocks";
    }
    return "unknown";
}

}  // extern "C"
