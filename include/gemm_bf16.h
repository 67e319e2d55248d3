/*
 * gemm_bf16.h -- C ABI of the GB300 (sm_103a) BF16 Tensor Core GEMM library
 * (libgemm_bf16.so).
 *
 * Operation (the pages' "Shape the operation", chapter 10 "Tensor Cores,
 * shapes, and tile alignment"; the mixed-precision paragraph of "The Tensor
 * Core" lesson):
 *
 *     C[M x N] = A[M x K] . B[K x N]
 *
 * with bf16 A and B, products accumulated in fp32 on the Tensor Cores, and C
 * written as fp32 or as bf16 (round to nearest even).  By default C is output
 * only: the "+ C" of D = A x B + C is taken with a zero C (the accumulator
 * starts at zero) and the previous contents of C are overwritten, never read;
 * the fused epilogue (gemm_epilogue_t) adds beta * C, bias and an activation.
 *
 * Conventions shared by every entry point
 *   - Dimensions are element counts; leading dimensions ("ld") are in
 *     elements, not bytes.  A row-major X[r][c] lives at X[r*ld + c]; a
 *     column-major one at X[c*ld + r].
 *   - Device pointers are raw CUDA device addresses.  The caller owns A, B, C
 *     and the stream and keeps them alive until the work on the stream has
 *     finished; the library never frees them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every launch is asynchronous on that stream; a return of
 *     GEMM_OK means the work was enqueued.  Faults found on the device (a
 *     pipeline wait that ran out of time) are reported by
 *     gemm_get_device_status().
 *   - Errors are returned as gemm_status_t; nothing here exits, aborts or
 *     prints.  Arguments are checked before any CUDA call is made.
 *
 * Alignment ("Record pointer alignment, leading dimensions, strides, and all
 * three contraction dimensions", chapter 10, "Padding efficiency"): the
 * operands are fed by TMA and stored with 16-byte vector stores, so
 *   - A, B and C start on a 16-byte boundary;
 *   - lda and ldb are multiples of 8 (16 bytes of bf16);
 *   - ldc is a multiple of 8 for bf16 C and of 4 for fp32 C.
 * M, N and K themselves need no particular multiple: ragged edges are
 * zero-filled on load and masked on store.  Nothing outside the M x N block
 * of C is written (columns N .. ldc-1 keep their contents, so C may be a
 * column slice of a wider matrix).  Each of M, N, K must be below 2^31.
 */
#ifndef GEMM_BF16_H
#define GEMM_BF16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;
typedef enum { GEMM_OUT_F32 = 0, GEMM_OUT_BF16 = 1 } gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,   /* negative or too large size, bad enum, short ld, NULL */
    GEMM_ERR_MISALIGNED = 2,      /* a pointer or leading dimension breaks the rules above */
    GEMM_ERR_NOT_SUPPORTED = 3,   /* a request the library cannot run (too many stream-K clusters;
                                     a convolution beyond an im2col box's range) */
    GEMM_ERR_NO_DEVICE = 4,       /* no usable CUDA device, or not an sm_103 part */
    GEMM_ERR_OUT_OF_MEMORY = 5,   /* the split-K workspace could not be grown */
    GEMM_ERR_LAUNCH = 6,          /* a CUDA runtime or driver call failed */
    GEMM_ERR_DEVICE_TIMEOUT = 7   /* a device-side pipeline wait ran out of time */
} gemm_status_t;

/* Kernel variants.  A tile is the block of C one work unit produces.
 *   1SM_128x256: one CTA per tile, tcgen05.mma.cta_group::1 with M = 128.
 *   1SM_128x128: the same with 128-column tiles (N = 128 per MMA), for a
 *     single row of tiles (M <= 128) with a long K: twice the work units of
 *     1SM_128x256, so the split that fills the SMs takes half the slices and
 *     half the fp32 partial bytes per CTA (see gemm_plan_for_device).
 *   2SM_256x256, 2SM_256x128: a cluster of two CTAs on a pair of SMs per
 *     tile, tcgen05.mma.cta_group::2 with M = 256; each CTA stages its own
 *     128 rows of A and half of the tile's columns of B, and holds its 128
 *     rows of the accumulator.
 * GEMM_KERNEL_AUTO lets the plan choose: both kernels spend the same time
 * on one k-tile of one tile, so it compares the k-tiles per resident cluster
 * with the work spread evenly, ceil(T k_tiles / C) (C = S single CTAs or S/2
 * pairs), and takes the single-CTA kernel only when that is under 93 % of
 * the pair kernel's (which keeps its tensor pipes about 7 % busier). */
typedef enum {
    GEMM_KERNEL_AUTO = 0,
    GEMM_KERNEL_1SM_128x256 = 1,
    GEMM_KERNEL_2SM_256x256 = 2,
    GEMM_KERNEL_2SM_256x128 = 3,
    GEMM_KERNEL_1SM_128x128 = 4
} gemm_kernel_variant_t;

/* Which resource sets the number of resident CTAs per SM. */
typedef enum {
    GEMM_LIMIT_REGISTERS = 0,
    GEMM_LIMIT_SMEM = 1,
    GEMM_LIMIT_TMEM = 2,
    GEMM_LIMIT_THREADS = 3,
    GEMM_LIMIT_BLOCKS = 4
} gemm_limiter_t;

/* Facts about one GPU that the plan depends on. */
typedef struct {
    int num_sms;                 /* S: streaming multiprocessors */
    int smem_per_sm;             /* bytes of shared memory per SM */
    int smem_optin_per_cta;      /* largest dynamic shared memory one CTA may request */
    int smem_reserved_per_cta;   /* bytes the runtime keeps per resident CTA */
    int regs_per_sm;             /* 32-bit registers per SM */
    int max_threads_per_sm;
    int max_ctas_per_sm;
    int tmem_cols_per_sm;        /* tensor-memory columns per SM (512 on sm_100-class parts) */
} gemm_device_desc_t;

/* Resource footprint of one CTA of a kernel. */
typedef struct {
    int regs_per_thread;         /* as compiled; 0 = unknown (registers then bind nothing) */
    int threads_per_cta;
    int smem_per_cta;            /* dynamic + static shared memory, bytes */
    int tmem_cols_per_cta;       /* tensor-memory columns allocated by one CTA */
    int cluster_size;            /* CTAs per cluster (1 or 2) */
    int max_active_clusters;     /* clusters resident at once on the device; 0 = unknown
                                    (then floor(S b / cluster_size)) */
} gemm_kernel_desc_t;

/*
 * The launch plan.  Closed forms from chapter 10, "Shape the operation" and
 * "Padding efficiency":
 *   grid      G = ceil(M/T_M) ceil(N/T_N) split_k        (split-K adds CTAs,
 *               "When shape alone can't fix wave efficiency")
 *   eta_wave    = G / (ceil(G / (S b)) S b)
 *   eta_pad     = M N K / (M' N' K'),  X' = ceil(X / T_X) T_X
 * and b, the CTAs per SM, from the tightest resource ("Grid 24 is not
 * headroom", "The question I never asked"): registers (per-thread count
 * rounded up to a multiple of 8, times the threads), shared memory (plus the
 * per-CTA reservation), tensor memory, threads, and the CTA limit.  eta_wave
 * is reported by that formula for both launch modes; a persistent launch
 * still runs ceil(G / (S b)) rounds of equal tiles.
 * For two-CTA tiles, G counts CTAs (two per tile and split) and S b is the
 * number of CTAs resident at once: resident clusters times two.
 */
typedef struct {
    int tile_m, tile_n, tile_k;  /* T_M x T_N x T_K of one tile */
    int stages;                  /* depth of the shared-memory operand ring */
    int threads_per_cta;
    int split_k;                 /* splits actually used (after auto choice and clamping) */
    int k_tiles;                 /* ceil(K / T_K) */
    int k_tiles_per_split;       /* largest k-tile count of one split */
    int num_sms;                 /* S */
    int ctas_per_sm;             /* b */
    int occupancy_limiter;       /* gemm_limiter_t */
    int persistent;              /* 1: grid = min(G, S b) CTAs looping over work units */
    int64_t tiles;               /* ceil(M/T_M) ceil(N/T_N) */
    int64_t grid;                /* G */
    int64_t launch_ctas;         /* CTAs actually launched for the main kernel */
    int64_t m_padded, n_padded, k_padded;  /* M', N', K' */
    double eta_wave;
    double eta_pad;
    double flops;                /* 2 M N K */
    int64_t smem_bytes;          /* dynamic shared memory per CTA of the main kernel */
    int64_t workspace_bytes;     /* fp32 partial tiles: split-K, split_k * tiles * tile_m * tile_n * 4;
                                    stream-K tail, one tile per resident cluster */
    int tmem_cols;               /* tensor-memory columns per CTA */
    int kernel_variant;          /* gemm_kernel_variant_t actually used */
    int cluster_size;            /* CTAs per tile */
    int64_t resident_ctas;       /* S b: CTAs resident at once */
    int64_t stream_k_tiles;      /* tiles whose k-iterations are spread over all clusters (0: none) */
    int64_t dp_tiles;            /* tiles computed whole, one cluster each */
    double eta_stream_k;         /* with a stream-K tail: ideal / actual per-cluster work
                                    (tiles*k_tiles/clusters over the largest share); 0 without */
    int raster_group_m;          /* m-tiles per raster group of the tile order: the option's value, or
                                    8 when the tiles make at least eight waves of the resident
                                    clusters on a persistent grid, else 16 */
} gemm_plan_t;

/* Elementwise work fused into the store of C (gemm_bf16_ex with
 * opts->epilogue != NULL), per output element:
 *
 *     C[m][n] := act(alpha * (A.B)[m][n] + beta * C[m][n] + bias[n])
 *
 * The Tensor Core's operation is D = A x B + C, and the work between the
 * matrix products -- activation functions, residual adds -- runs on the
 * ordinary lanes (lesson "The Tensor Core", its opening and the paragraph on
 * what work the Tensor Cores speed up): here the epilogue threads do it on
 * the fp32 accumulator before the single rounding to C's type.  The pages name
 * no particular activation; these are offered:
 *   GEMM_ACT_NONE  x
 *   GEMM_ACT_RELU  max(x, 0)
 *   GEMM_ACT_GELU  x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)), the erf form
 * The sum and the activation are evaluated in fp32 in the order written
 * (alpha * acc, then + beta * C, then + bias).  On the device erfc is the
 * rational approximation of Abramowitz & Stegun 7.1.26 (absolute error at
 * most 1.5e-7), so GELU is within 2^-20 |x| of x * Phi(x) before rounding.  C is read in place before it
 * is overwritten (only when beta != 0); bias is NULL or a device array of N
 * fp32 values on a 16-byte boundary.  With K == 0 the product is zero and
 * C := act(beta * C + bias).  Split-K applies it in the combine kernel after
 * the slices are added; a stream-K tile after its partial sums are added. */
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU = 2 } gemm_activation_t;

typedef struct {
    float alpha;                 /* scale of A.B */
    float beta;                  /* scale of the previous C; 0: C is not read */
    const float *bias;           /* N fp32 values added per column, or NULL */
    int activation;              /* gemm_activation_t */
} gemm_epilogue_t;

/* Options of gemm_bf16_ex.  Zero-initialise and set what you need. */
typedef struct {
    int split_k;                 /* 0: the plan chooses; 1: off; >1: clamped to [1, k_tiles] */
    int non_persistent;          /* 1: one CTA per work unit (grid G) instead of a persistent grid */
    int raster_group_m;          /* m-tiles per raster group for L2 reuse; 0: default (8 when the tiles
                                    make at least eight waves of the resident clusters, else 16) */
    void *mainloop_done_event;   /* cudaEvent_t or NULL: recorded on the stream after the main
                                    kernel, before the split-K combine kernel */
    int timeout_ms;              /* per-wait device time limit; 0: default (4000 ms plus 8 us for
                                    each k-tile of the longest work unit and stream-K range) */
    int debug_skip_load;         /* test hook; must be 0 in normal use.  k: the producer leaves
                                    the k-th stage load (1-based, counting from the first load of
                                    CTA 0) unissued, so its consumer's wait runs out and the call
                                    ends with GEMM_ERR_DEVICE_TIMEOUT on the device */
    int kernel_variant;          /* gemm_kernel_variant_t; 0 = the plan chooses */
    int no_stream_k;             /* 0: the plan decides on a stream-K tail (see gemm_plan_for_device);
                                    1: never spread tiles over the clusters (stream-K);
                                   -1: always, whenever the tile count is not a multiple of the
                                       resident clusters (all tiles below two waves) */
    const gemm_epilogue_t *epilogue;   /* NULL: C = A.B; else the fused epilogue above (read
                                          during the call, not kept) */
} gemm_options_t;

/* Fill `dev` with the facts of CUDA device `device`. */
gemm_status_t gemm_device_desc_query(int device, gemm_device_desc_t *dev);

/* The footprint of one kernel variant (GEMM_KERNEL_AUTO: the variant the
 * plan chooses by default).  Registers and resident clusters come from the
 * compiled kernel on the current device when there is one, else 0. */
gemm_status_t gemm_kernel_desc(int kernel_variant, gemm_kernel_desc_t *kern);

/* Resident CTAs per SM for a footprint on a device (host arithmetic only).
 * Returns INVALID_VALUE for non-positive threads or a footprint that fits
 * zero times (then *ctas_per_sm is 0). */
gemm_status_t gemm_occupancy(const gemm_kernel_desc_t *kern, const gemm_device_desc_t *dev,
                             int *ctas_per_sm, int *limiter);

/*
 * Plan a GEMM for explicit device and kernel facts; host arithmetic only, no
 * CUDA call.  Same argument rules as gemm_bf16_ex (opts may be NULL); `kern`
 * describes the footprint of the variant opts selects (GEMM_KERNEL_AUTO
 * resolves to the default variant).
 *
 * Work decomposition, in order (T tiles, C resident clusters):
 *   - split_k > 1: split-K as asked (clamped to the k-tile count);
 *   - split_k = 0, a persistent launch, no_stream_k <= 0, T not a multiple of
 *     C, and either no_stream_k < 0 or (T >= C and the partly filled last
 *     wave leaves, per cluster on average, at least 12 k-tiles of 128 of a
 *     128 x 256 block per SM idle): a stream-K tail -- the last C + (T mod C)
 *     tiles (all T when T < 2C) have their k-iterations dealt out evenly over
 *     the C clusters in contiguous ranges, the rest are computed whole; with a
 *     GELU epilogue or one that reads C the ranges are made of whole half
 *     tiles when k_tiles is even and at least 8, else a range boundary within
 *     k_tiles / 4 of a tile's edge moves to the edge (a long epilogue should
 *     not follow a few k-tiles of MMAs);
 *   - split_k = 0, and T * 8 <= C with K >= 2048 or T * 4 <= C with
 *     K >= 6144: split-K chosen by the plan (C / T slices, each at least 4
 *     k-tiles long);
 *   - otherwise one cluster per tile.
 * With the plan's own variant, a small GEMM (256 x 128 pair tiles filling at
 * most half the resident pairs, K < 2048) runs on the 256 x 128 pair kernel.
 * A single row of tiles (M <= 128, N > 128) with K >= 2048 runs on the
 * 128 x 128 single-CTA kernel when its work units (tiles times the split
 * asked for, or the plan's own split for those tiles) fit in one wave and an
 * estimate of its time beats the 128 x 256 plan's: the operand bytes one CTA
 * streams at about 100 GB/s per SM, at least the unique operand bytes at
 * about 6.8 TB/s, plus, with split-K, about 6 us and the fp32 partial bytes
 * at about 2 TB/s; within 0.5 us the plan with more work units wins.
 * Handing partial tiles between CTAs costs a roughly fixed few to 25 us on
 * GB300 (fp32 partials through L2 and a fix-up or a combine kernel), so the
 * plan spreads or splits the work only where the longer K repays it.
 */
gemm_status_t gemm_plan_for_device(int64_t M, int64_t N, int64_t K,
                                   gemm_layout_t layout_a, gemm_layout_t layout_b,
                                   gemm_dtype_t out_dtype, const gemm_options_t *opts,
                                   const gemm_device_desc_t *dev,
                                   const gemm_kernel_desc_t *kern, gemm_plan_t *plan);

/* Plan a GEMM on the current CUDA device exactly as gemm_bf16_ex would run it. */
gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K,
                        gemm_layout_t layout_a, gemm_layout_t layout_b,
                        gemm_dtype_t out_dtype, const gemm_options_t *opts, gemm_plan_t *plan);

/*
 * C = A . B on `stream`.
 *   A: M x K bf16, GEMM_ROW_MAJOR (lda >= K) or GEMM_COL_MAJOR (lda >= M,
 *      i.e. stored as K rows of M contiguous values).
 *   B: K x N bf16, GEMM_COL_MAJOR (ldb >= K, i.e. stored as N rows of K
 *      contiguous values) or GEMM_ROW_MAJOR (ldb >= N).
 *   C: M x N row-major (ldc >= N), fp32 or bf16 per out_dtype.
 *   All four layout pairs run the same kernels: an operand whose K is
 *   contiguous is staged K-major, the others M- or N-major, and the Tensor
 *   Core reads either form from shared memory (the transpose bits of the
 *   instruction descriptor).
 *   split_k: 0 = the plan chooses, 1 = off, > 1 = that many K slices
 *      (clamped to the k-tile count).  With more than one slice the partial
 *      sums go to an fp32 workspace owned by the library and a second kernel
 *      adds them in slice order 0, 1, ... and writes C.
 * M == 0 or N == 0 is a no-op; K == 0 writes zeros to C.
 * The split-K workspace grows on demand with cudaMalloc (a synchronising
 * call); reserve it beforehand with gemm_reserve_workspace() to keep
 * allocation out of timed regions and stream captures.
 * Calls that share the workspace must not overlap in time on different
 * streams of one device.  The library's host-side bookkeeping is
 * thread-safe: while one host thread enqueues work that reads the workspace,
 * a lock keeps every other thread from growing or freeing it.  Work enqueued
 * by several host threads must still not overlap on the GPU, as above.
 */
gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K,
                        const void *A, int64_t lda, const void *B, int64_t ldb,
                        void *C, int64_t ldc,
                        gemm_layout_t layout_a, gemm_layout_t layout_b,
                        gemm_dtype_t out_dtype, int split_k, void *stream);

/*
 * gemm_bf16_splitk_noalloc -- gemm_bf16 for callers that must not allocate
 * device memory.  The pages have no counterpart to this entry point; it is
 * the library's own.
 *
 * Who needs it: gemm_bf16 grows its split-K workspace with cudaMalloc the
 * first time a large enough split is asked for.  Some callers cannot allow
 * that -- a process whose device memory is handed out entirely by its own
 * pool allocator (a raw cudaMalloc would fail, or carve memory out from under
 * the pool), a long-running service that keeps a fixed memory footprint and
 * must never meet an out-of-memory error in the middle of its work, or a
 * latency-critical loop that cannot absorb cudaMalloc's implicit
 * synchronisation of the whole device.  This entry point keeps the fp32
 * partial sums in a fixed array compiled into the library instead
 * (GEMM_NOALLOC_SCRATCH_BYTES = 16 MiB), which every GPU that loads the
 * library holds until the process exits.  It calls no cudaMalloc, cudaFree
 * or other allocating routine.
 *
 * Arguments, layouts, alignment rules and results are those of gemm_bf16.
 * The split actually used (split_k, or the plan's choice when split_k is 0)
 * must satisfy  split * tiles * tile_m * tile_n <= GEMM_NOALLOC_SCRATCH_FLOATS,
 * counting whole (padded) tiles of the kernel the plan picks; that is the
 * workspace_bytes / 4 of gemm_plan with the same split_k and no_stream_k = 1
 * (with 128 x 256 tiles and M, N multiples of them it is split * M * N);
 * otherwise the call returns GEMM_ERR_INVALID_VALUE and launches nothing.
 * split_k = 1 uses no scratch at all, and this entry point never uses a
 * stream-K tail.
 *
 * The first call on a device looks up the array's address on that device
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call shares the one array, and the array keeps whatever the last
 * call left in it.  Nothing needs clearing: each partial sum a call reads was
 * written earlier by the same call.  Calls whose work can overlap on the GPU
 * (other streams, other host threads) race on the array and must be
 * serialised by the caller.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
#define GEMM_NOALLOC_SCRATCH_FLOATS (GEMM_NOALLOC_SCRATCH_BYTES / 4u)
gemm_status_t gemm_bf16_splitk_noalloc(int64_t M, int64_t N, int64_t K,
                                       const void *A, int64_t lda, const void *B, int64_t ldb,
                                       void *C, int64_t ldc,
                                       gemm_layout_t layout_a, gemm_layout_t layout_b,
                                       gemm_dtype_t out_dtype, int split_k, void *stream);

/* gemm_bf16 with options (launch mode, raster group, timing event, device
 * time limit, kernel variant, stream-K).  opts == NULL behaves as gemm_bf16
 * with split_k = 0.  A stream-K tail keeps fp32 partial tiles in the library's
 * workspace and hands them between the resident clusters of one launch
 * through flags in device memory; like split-K, calls that share the
 * workspace must not overlap in time. */
gemm_status_t gemm_bf16_ex(int64_t M, int64_t N, int64_t K,
                           const void *A, int64_t lda, const void *B, int64_t ldb,
                           void *C, int64_t ldc,
                           gemm_layout_t layout_a, gemm_layout_t layout_b,
                           gemm_dtype_t out_dtype, const gemm_options_t *opts, void *stream);

/*
 * 2-D convolution (forward) as an implicit GEMM.
 *
 * Convolutions reach the Tensor Cores through im2col / implicit GEMM (lesson
 * "The Tensor Core", the paragraph on what work the Tensor Cores speed up):
 *
 *   y[n][p][q][k] = sum over r < R, s < S, c < C of
 *                   x[n][p*stride_h - pad_h + r*dil_h][q*stride_w - pad_w + s*dil_w][c] * w[k][r][s][c]
 *
 * with x zero outside the image (the padding).  It is the GEMM
 * C (N P Q x K) = A (N P Q x R S C) . B (R S C x K) in which row m of A is the
 * receptive field of output pixel m -- never formed in memory: TMA's im2col
 * mode loads each A box (128 output pixels x 64 channels at one filter tap)
 * straight from x, zero-filling the padding.  P and Q are
 * (H + 2 pad - dil (R - 1) - 1) / stride + 1 (integer division, >= 1).
 *
 *   x: N x H x W x C bf16, NHWC, dense.       w: K x R x S x C bf16, KRSC, dense.
 *   y: N x P x Q x K, dense (row m = (n P + p) Q + q of an N P Q x K
 *      row-major matrix), fp32 or bf16 per out_dtype.
 * Requirements: every size >= 1, strides and dilations >= 1, paddings >= 0;
 * C a multiple of 8 (16-byte pixel rows); K a multiple of 8 for bf16 y or 4
 * for fp32 y; x, w, y on 16-byte boundaries (GEMM_ERR_MISALIGNED otherwise);
 * N P Q and R S C below 2^31; paddings and dil (R - 1), dil (S - 1) at most
 * 127 (GEMM_ERR_NOT_SUPPORTED beyond: the range of an im2col pixel box).  The
 * options work as for gemm_bf16_ex (kernel variant, split-K, stream-K, the
 * fused epilogue -- a bias per output channel k).
 */
typedef struct {
    int64_t N, H, W, C;          /* input */
    int64_t K, R, S;             /* filter: K output channels of R x S taps */
    int pad_h, pad_w;
    int stride_h, stride_w;
    int dil_h, dil_w;
} gemm_conv2d_desc_t;

/* The output extent P x Q of `d`; GEMM_ERR_INVALID_VALUE if it is empty or a
 * field is out of range. */
gemm_status_t gemm_conv2d_out_dims(const gemm_conv2d_desc_t *d, int64_t *P, int64_t *Q);

/* The plan of the implicit GEMM (M = N P Q, N = K, K = R S C rounded up to
 * whole 64-channel blocks per tap) on the current device. */
gemm_status_t gemm_conv2d_plan(const gemm_conv2d_desc_t *d, gemm_dtype_t out_dtype, const gemm_options_t *opts,
                               gemm_plan_t *plan);

/* y = conv2d(x, w) on `stream` (opts may be NULL). */
gemm_status_t gemm_conv2d_fprop_bf16(const gemm_conv2d_desc_t *d, const void *x, const void *w, void *y,
                                     gemm_dtype_t out_dtype, const gemm_options_t *opts, void *stream);

/*
 * Host-resident GEMMs, copies overlapped with the Tensor Core work.
 *
 * The pages measure the kernel on operands already in device memory; a caller
 * whose matrices live in host memory also pays the copies over the host link,
 * which for a 4096^3 problem take several times longer than the product.
 * gemm_bf16_host_batch runs `count` independent problems whose A, B and C are
 * HOST pointers.  Each problem's operands are copied into one of two device
 * staging slots, the product is computed there by the kernels of gemm_bf16_ex,
 * and C is copied back -- every problem moves its own bytes both ways -- but
 * the library overlaps problem i's result copy and problem i+1's operand
 * copies with the products on three streams of its own (operand copies,
 * products, result copies).
 *
 *   problems[i]: sizes, layouts and leading dimensions as for gemm_bf16
 *      (lda, ldb, ldc in elements of the host arrays; no alignment rule on the
 *      host side: the staging copies are pitched to 16-byte rows on the
 *      device, so any M, N, K are accepted).
 *   out_dtype, opts: as for gemm_bf16_ex, applied to every problem; an
 *      epilogue's bias stays a DEVICE array.  With an epilogue whose beta is
 *      non-zero, C is also copied in before the product.
 *   stream: the copies of problem 0 start after the work enqueued on `stream`
 *      before the call, and `stream` waits for the last result copy, so a
 *      cudaStreamSynchronize(stream) later means every C is in host memory.
 *      The call itself returns once everything is enqueued: the host arrays
 *      must stay valid and unchanged until then.
 * Pinned host memory (cudaHostAlloc or cudaHostRegister) is needed for the
 * copies to be asynchronous and to overlap; pageable memory gives the same
 * results, with copies the CUDA runtime serialises through its own buffers.
 * All problems are checked before anything is enqueued (INVALID_VALUE: a NULL
 * pointer, a leading dimension below its minimum, a bad size, layout, type or
 * option).  The staging slots grow on demand with cudaMalloc (synchronising
 * the library's streams first); gemm_release_workspace frees them.  Calls on
 * one device are serialised by a lock; the products share the split-K
 * workspace with the other entry points, as usual. */
typedef struct {
    int64_t M, N, K;
    const void *A;               /* host */
    int64_t lda;
    gemm_layout_t layout_a;
    const void *B;               /* host */
    int64_t ldb;
    gemm_layout_t layout_b;
    void *C;                     /* host, M x N row-major */
    int64_t ldc;
} gemm_host_problem_t;

gemm_status_t gemm_bf16_host_batch(int64_t count, const gemm_host_problem_t *problems,
                                   gemm_dtype_t out_dtype, const gemm_options_t *opts, void *stream);

/* Grow the current device's split-K workspace to at least `bytes`. */
gemm_status_t gemm_reserve_workspace(size_t bytes);

/* Free the split-K workspaces and the host-batch staging slots of every
 * device (waits for each device first). */
void gemm_release_workspace(void);

/*
 * Synchronise `stream`, then report and clear the current device's fault
 * word: GEMM_OK, GEMM_ERR_DEVICE_TIMEOUT (a pipeline wait ran out of time;
 * if `where` is not NULL it receives the bit set of the waits that gave up:
 * 1 producer slot wait, 2 MMA operand wait, 4 MMA accumulator wait,
 * 8 epilogue accumulator wait, 16 end-of-kernel drain, 32 stream-K partial
 * hand-off, 64 fused epilogue's load of the previous C), or GEMM_ERR_LAUNCH
 * if the synchronisation itself failed.
 */
gemm_status_t gemm_get_device_status(void *stream, unsigned int *where);

/* A static, human-readable name for a status code. */
const char *gemm_status_string(gemm_status_t status);

/* Name of a gemm_limiter_t value ("registers", "smem", "tmem", "threads", "blocks"). */
const char *gemm_limiter_string(int limiter);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_BF16_H */
