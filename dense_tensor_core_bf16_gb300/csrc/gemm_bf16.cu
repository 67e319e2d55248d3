// gemm_bf16.cu -- BF16 Tensor Core GEMM for GB300 (sm_103a): kernels and the
// C-ABI launcher.  Contract: include/gemm_bf16.h.
//
// Method (chapter 10 "Tensor Cores, shapes, and tile alignment"; lesson
// "The Tensor Core"; post "Grid 24 is not headroom"):
//   * two-sided tiling: A and B tiles are staged once in shared memory and
//     reused by every MMA of the tile ("feeding it is the hard part");
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

enum : unsigned { SITE_PRODUCER = 1u, SITE_MMA_OPERANDS = 2u, SITE_MMA_ACC = 4u, SITE_EPI_ACC = 8u, SITE_DRAIN = 16u };

struct KernelParams {
    int M, N, K;
    int tiles_m, tiles_n;
    int k_tiles;                 // ceil(K / TILE_K)
    int split_k;
    int group_m;                 // m-tiles per raster group
    long long num_units;         // tiles * split_k
    void *out;                   // C, or the fp32 partial buffer when split_k > 1
    long long ld_out;            // leading dimension of `out`, elements
    long long split_stride;      // elements between consecutive partial slices
    int out_bf16;                // 1: bf16 stores, 0: fp32 stores
    unsigned long long timeout_ns;
    int skip_load;               // test hook (0 = off)
};

// Barrier indices in shared memory.
constexpr int BAR_FULL = 0;                          // [STAGES] operands landed
constexpr int BAR_EMPTY = STAGES;                    // [STAGES] slot free again
constexpr int BAR_ACC_FULL = 2 * STAGES;             // [ACC_BUFS] accumulator complete
constexpr int BAR_ACC_EMPTY = 2 * STAGES + ACC_BUFS; // [ACC_BUFS] accumulator drained
constexpr int BAR_DRAIN = 2 * STAGES + 2 * ACC_BUFS; // all MMAs of this CTA done

// Wait for the phase of `bar` with parity `parity`.  Gives up after
// `timeout_ns` (recording `site` in the fault word and raising the CTA's abort
// flag), or -- when `honor_abort` -- as soon as another role has given up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           unsigned long long timeout_ns, unsigned site, bool honor_abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
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

struct Unit {
    int tm, tn;         // tile coordinates (in tiles)
    int split;          // K slice
    int kb_begin;       // first k-tile of the slice
    int kb_count;       // k-tiles in the slice (>= 1)
};

// Work unit u -> tile and K slice.  Tiles are visited in groups of group_m
// tile-rows, column by column inside a group, so that the CTAs resident at
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
    return w;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Store 32 consecutive fp32 accumulator values of one row, columns col0..col0+31.
__device__ __forceinline__ void store_row_chunk(const KernelParams &p, const Unit &w, int row, int col0,
                                                const uint32_t (&r)[32]) {
    if (p.out_bf16) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) + static_cast<long long>(row) * p.ld_out + col0;
        if (col0 + 32 <= p.N) {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                d4[v] = make_uint4(pack_bf16x2(r[8 * v + 0], r[8 * v + 1]), pack_bf16x2(r[8 * v + 2], r[8 * v + 3]),
                                   pack_bf16x2(r[8 * v + 4], r[8 * v + 5]), pack_bf16x2(r[8 * v + 6], r[8 * v + 7]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (col0 + j < p.N) dst[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
            }
        }
    } else {
        float *dst = static_cast<float *>(p.out) + static_cast<long long>(w.split) * p.split_stride +
                     static_cast<long long>(row) * p.ld_out + col0;
        if (col0 + 32 <= p.N) {
            float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                d4[v] = make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                    __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (col0 + j < p.N) dst[j] = __uint_as_float(r[j]);
            }
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_bf16_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             const KernelParams p) {
    extern __shared__ uint8_t smem_raw[];
    // Operand tiles must start on the 1024-byte swizzle-atom boundary.
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sA = ptx::smem_addr(smem);                      // STAGES A tiles
    const uint32_t sB = sA + STAGES * A_STAGE_BYTES;               // STAGES B tiles
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARRIERS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto bar = [bar0](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);    // producer's arrive + TMA bytes
            ptx::mbar_init(bar(BAR_EMPTY + s), 1);   // MMA commit
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            ptx::mbar_init(bar(BAR_ACC_FULL + b), 1);              // MMA commit
            ptx::mbar_init(bar(BAR_ACC_EMPTY + b), EPI_THREADS);   // every epilogue thread
        }
        ptx::mbar_init(bar(BAR_DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_a);
        ptx::prefetch_tensormap(&tmap_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish_alloc_permit();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

    if (warp == 0) {
        // ---------------- producer: TMA copies into the ring ----------------
        if (lane == 0) {
            uint32_t it = 0, issued = 0;
            bool ok = true;
            for (long long u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
                const Unit w = decode_unit(u, p);
                for (int kb = 0; kb < w.kb_count; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_phase(bar(BAR_EMPTY + s), ph ^ 1u, abort_flag, p.timeout_ns, SITE_PRODUCER, true)) {
                        ok = false;
                        break;
                    }
                    ++issued;
                    if (p.skip_load != 0 && blockIdx.x == 0 && issued == static_cast<uint32_t>(p.skip_load)) {
                        continue;   // test hook: this slot is never filled
                    }
                    ptx::mbar_arrive_expect_tx(bar(BAR_FULL + s), STAGE_BYTES);
                    const int kc = (w.kb_begin + kb) * TILE_K;
                    ptx::tma_load_2d(sA + s * A_STAGE_BYTES, &tmap_a, bar(BAR_FULL + s), kc, w.tm * TILE_M);
                    ptx::tma_load_2d(sB + s * B_STAGE_BYTES, &tmap_b, bar(BAR_FULL + s), kc, w.tn * TILE_N);
                }
            }
            // No copy may still be writing this CTA's shared memory when it
            // exits: wait (bounded) for the last STAGES loads.  Earlier ones
            // were consumed by the MMA warp before their slots were reused.
            const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
            for (uint32_t j = first; j < it; ++j) {
                wait_phase(bar(BAR_FULL + j % STAGES), (j / STAGES) & 1u, abort_flag, p.timeout_ns, SITE_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: one thread drives the Tensor Core ------
        if (lane == 0) {
            constexpr uint32_t IDESC = ptx::idesc_bf16_f32(TILE_M, TILE_N);
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (long long u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++tc) {
                const Unit w = decode_unit(u, p);
                const uint32_t buf = tc & 1u;
                const uint32_t use = tc >> 1;
                if (!wait_phase(bar(BAR_ACC_EMPTY + buf), (use & 1u) ^ 1u, abort_flag, p.timeout_ns, SITE_MMA_ACC,
                                true)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * TILE_N;
                for (int kb = 0; kb < w.kb_count; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_phase(bar(BAR_FULL + s), ph, abort_flag, p.timeout_ns, SITE_MMA_OPERANDS, true)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint64_t a_desc = ptx::smem_desc_kmajor_sw128(sA + s * A_STAGE_BYTES);
                    const uint64_t b_desc = ptx::smem_desc_kmajor_sw128(sB + s * B_STAGE_BYTES);
#pragma unroll
                    for (int k = 0; k < TILE_K / MMA_K; ++k) {
                        // next 16 elements of K: +32 bytes inside the swizzled
                        // 128-byte row, i.e. +2 in the address>>4 field
                        ptx::mma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, IDESC, (kb | k) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(BAR_EMPTY + s));   // slot reusable once these MMAs have read it
                }
                if (!ok) break;
                ptx::mma_commit(bar(BAR_ACC_FULL + buf));  // accumulator complete
            }
            // Every MMA issued here must finish before TMEM is released.
            ptx::mma_commit(bar(BAR_DRAIN));
            wait_phase(bar(BAR_DRAIN), 0, abort_flag, p.timeout_ns, SITE_DRAIN, false);
        }
    } else {
        // ---------------- epilogue: TMEM -> registers -> global ---------------
        const int quarter = warp & 3;            // TMEM lanes this warp may read: 32*quarter ..
        const int row_in_tile = quarter * 32 + lane;
        uint32_t tc = 0;
        for (long long u = blockIdx.x; u < p.num_units; u += gridDim.x, ++tc) {
            const Unit w = decode_unit(u, p);
            const uint32_t buf = tc & 1u;
            const uint32_t use = tc >> 1;
            const bool ok = wait_phase(bar(BAR_ACC_FULL + buf), use & 1u, abort_flag, p.timeout_ns, SITE_EPI_ACC, true);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after_sync();
            const int row = w.tm * TILE_M + row_in_tile;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * TILE_N;
            const int col_base = w.tn * TILE_N;
#pragma unroll 1
            for (int c = 0; c < TILE_N / 32; ++c) {
                const int col0 = col_base + c * 32;
                if (col0 >= p.N) break;          // same for the whole warp
                uint32_t r[32];
                __syncwarp();
                ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
                ptx::tmem_wait_ld();
                if (row < p.M) store_row_chunk(p, w, row, col0, r);
            }
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar(BAR_ACC_EMPTY + buf));
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// C[m][n] = sum over s = 0, 1, ..., split-1 of P[s][m][n], in that order, then
// cast to the output type.  One thread per 4 consecutive columns of a row.
__global__ void __launch_bounds__(256)
    splitk_combine_kernel(const float *__restrict__ part, long long ldp, long long split_stride, int split, int M,
                          int N, void *C, long long ldc, int out_bf16) {
    const long long n4 = (N + 3) / 4;
    const long long total = static_cast<long long>(M) * n4;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int m = static_cast<int>(idx / n4);
        const int col = static_cast<int>(idx - static_cast<long long>(m) * n4) * 4;
        const float *src = part + static_cast<long long>(m) * ldp + col;
        float4 acc = __ldcs(reinterpret_cast<const float4 *>(src));
#pragma unroll 8
        for (int s = 1; s < split; ++s) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(src + s * split_stride));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float a[4] = {acc.x, acc.y, acc.z, acc.w};
        if (out_bf16) {
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(C) + static_cast<long long>(m) * ldc + col;
            if (col + 4 <= N) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(a[0], a[1]);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(a[2], a[3]);
                uint2 v;
                v.x = *reinterpret_cast<const uint32_t *>(&lo);
                v.y = *reinterpret_cast<const uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(dst) = v;
            } else {
                for (int j = 0; j < 4 && col + j < N; ++j) dst[j] = __float2bfloat16_rn(a[j]);
            }
        } else {
            float *dst = static_cast<float *>(C) + static_cast<long long>(m) * ldc + col;
            if (col + 4 <= N) {
                *reinterpret_cast<float4 *>(dst) = acc;
            } else {
                for (int j = 0; j < 4 && col + j < N; ++j) dst[j] = a[j];
            }
        }
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

// ------------------------------------------------------------------ host side

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    gemm_device_desc_t desc{};
    int regs_per_thread = 0;
    float *workspace = nullptr;
    size_t workspace_bytes = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

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
        if (cudaFuncSetAttribute(gemm_bf16_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, gemm_bf16_tcgen05_kernel) != cudaSuccess) return GEMM_ERR_LAUNCH;
        ds.regs_per_thread = fa.numRegs;
        if (!g_encode_tiled) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult qr{};
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
                    cudaSuccess ||
                qr != cudaDriverEntryPointSuccess || fn == nullptr)
                return GEMM_ERR_LAUNCH;
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        ds.ready = true;
    }
    *out = &ds;
    return GEMM_OK;
}

gemm_kernel_desc_t main_kernel_desc(int regs_per_thread) {
    gemm_kernel_desc_t k{};
    k.regs_per_thread = regs_per_thread;
    k.threads_per_cta = NUM_THREADS;
    k.smem_per_cta = SMEM_BYTES;
    k.tmem_cols_per_cta = TMEM_COLS;
    return k;
}

// A K-major bf16 operand with `rows` rows of `k` elements, `ld` apart.
gemm_status_t encode_operand(CUtensorMap *map, const void *ptr, int64_t k, int64_t rows, int64_t ld, int box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(TILE_K), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t elem_strides[2] = {1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                                elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

gemm_status_t ensure_workspace(int device, DeviceState &ds, size_t bytes) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ds.workspace_bytes >= bytes) return GEMM_OK;
    if (ds.workspace) {
        cudaDeviceSynchronize();   // the old buffer may still be read by queued work
        cudaFree(ds.workspace);
        ds.workspace = nullptr;
        ds.workspace_bytes = 0;
    }
    (void)device;
    void *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_OUT_OF_MEMORY;
    }
    ds.workspace = static_cast<float *>(p);
    ds.workspace_bytes = bytes;
    return GEMM_OK;
}

gemm_status_t launch_fill_zero(int64_t M, int64_t N, void *C, int64_t ldc, int esize, int num_sms,
                               cudaStream_t stream) {
    const long long total = M * N;
    long long blocks = (total + 255) / 256;
    if (blocks > 4LL * num_sms) blocks = 4LL * num_sms;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, fill_zero_kernel, C, static_cast<long long>(ldc), static_cast<int>(M),
                              static_cast<int>(N), esize) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_LAUNCH;
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

gemm_status_t gemm_kernel_desc(gemm_kernel_desc_t *kern) {
    if (!kern) return GEMM_ERR_INVALID_VALUE;
    int regs = 0;
    int device = 0;
    if (cudaGetDevice(&device) == cudaSuccess) {
        DeviceState *ds = nullptr;
        if (device_state(device, &ds) == GEMM_OK) regs = ds->regs_per_thread;
    }
    cudaGetLastError();
    *kern = main_kernel_desc(regs);
    return GEMM_OK;
}

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, gemm_layout_t layout_a, gemm_layout_t layout_b,
                        gemm_dtype_t out_dtype, int split_k, gemm_plan_t *plan) {
    if (!plan) return GEMM_ERR_INVALID_VALUE;
    gemm_status_t st = check_problem(M, N, K, layout_a, layout_b, out_dtype, split_k);
    if (st != GEMM_OK) return st;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    DeviceState *ds = nullptr;
    st = device_state(device, &ds);
    if (st != GEMM_OK) return st;
    return make_plan(M, N, K, layout_a, layout_b, out_dtype, split_k, 1, ds->desc, main_kernel_desc(ds->regs_per_thread),
                     plan);
}

gemm_status_t gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                           void *C, int64_t ldc, gemm_layout_t layout_a, gemm_layout_t layout_b,
                           gemm_dtype_t out_dtype, const gemm_options_t *opts, void *stream) {
    gemm_options_t o{};
    if (opts) o = *opts;
    gemm_status_t st = check_problem(M, N, K, layout_a, layout_b, out_dtype, o.split_k);
    if (st != GEMM_OK) return st;
    if (o.timeout_ms < 0 || o.raster_group_m < 0 || o.debug_skip_load < 0) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_OK;
    const int esize = out_dtype == GEMM_OUT_BF16 ? 2 : 4;
    if (!C || ldc < N) return GEMM_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(C) % 16 != 0 || (ldc * esize) % 16 != 0) return GEMM_ERR_MISALIGNED;
    if (K > 0) {
        if (!A || !B || lda < K || ldb < K) return GEMM_ERR_INVALID_VALUE;
        if (reinterpret_cast<uintptr_t>(A) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0 || lda % 8 != 0 ||
            ldb % 8 != 0)
            return GEMM_ERR_MISALIGNED;
    }

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    DeviceState *ds = nullptr;
    st = device_state(device, &ds);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (K == 0) return launch_fill_zero(M, N, C, ldc, esize, ds->desc.num_sms, s);

    gemm_plan_t plan;
    st = make_plan(M, N, K, layout_a, layout_b, out_dtype, o.split_k, o.non_persistent ? 0 : 1, ds->desc,
                   main_kernel_desc(ds->regs_per_thread), &plan);
    if (st != GEMM_OK) return st;
    const int64_t ldp = (N + 3) / 4 * 4;
    if (plan.split_k > 1) {
        st = ensure_workspace(device, *ds, static_cast<size_t>(plan.workspace_bytes));
        if (st != GEMM_OK) return st;
    }

    CUtensorMap tmap_a, tmap_b;
    st = encode_operand(&tmap_a, A, K, M, lda, TILE_M);
    if (st != GEMM_OK) return st;
    st = encode_operand(&tmap_b, B, K, N, ldb, TILE_N);
    if (st != GEMM_OK) return st;

    KernelParams p{};
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((M + TILE_M - 1) / TILE_M);
    p.tiles_n = static_cast<int>((N + TILE_N - 1) / TILE_N);
    p.k_tiles = plan.k_tiles;
    p.split_k = plan.split_k;
    p.group_m = o.raster_group_m > 0 ? o.raster_group_m : DEFAULT_RASTER_GROUP_M;
    p.num_units = plan.grid;
    if (plan.split_k > 1) {
        p.out = ds->workspace;
        p.ld_out = ldp;
        p.split_stride = M * ldp;
        p.out_bf16 = 0;
    } else {
        p.out = C;
        p.ld_out = ldc;
        p.split_stride = 0;
        p.out_bf16 = out_dtype == GEMM_OUT_BF16 ? 1 : 0;
    }
    const int timeout_ms = o.timeout_ms > 0 ? o.timeout_ms : DEFAULT_TIMEOUT_MS;
    p.timeout_ns = static_cast<unsigned long long>(timeout_ms) * 1000000ull;
    p.skip_load = o.debug_skip_load;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.launch_ctas));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    if (cudaLaunchKernelEx(&cfg, gemm_bf16_tcgen05_kernel, tmap_a, tmap_b, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (o.mainloop_done_event && cudaEventRecord(static_cast<cudaEvent_t>(o.mainloop_done_event), s) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    if (plan.split_k > 1) {
        const long long total = M * ((N + 3) / 4);
        long long blocks = (total + 255) / 256;
        const long long cap = 4LL * ds->desc.num_sms;
        if (blocks > cap) blocks = cap;
        cudaLaunchConfig_t cc{};
        cc.gridDim = dim3(static_cast<unsigned>(blocks));
        cc.blockDim = dim3(256);
        cc.stream = s;
        if (cudaLaunchKernelEx(&cc, splitk_combine_kernel, static_cast<const float *>(ds->workspace),
                               static_cast<long long>(ldp), static_cast<long long>(M * ldp), plan.split_k,
                               static_cast<int>(M), static_cast<int>(N), C, static_cast<long long>(ldc),
                               out_dtype == GEMM_OUT_BF16 ? 1 : 0) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    }
    return GEMM_OK;
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
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    DeviceState *ds = nullptr;
    gemm_status_t st = device_state(device, &ds);
    if (st != GEMM_OK) return st;
    return ensure_workspace(device, *ds, bytes);
}

void gemm_release_workspace(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int current = -1;
    if (cudaGetDevice(&current) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    for (int d = 0; d < kMaxDevices; ++d) {
        DeviceState &ds = g_devices[d];
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
    const int esize = out_dtype == GEMM_OUT_BF16 ? 2 : 4;
    if (!C || ldc < N) return GEMM_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(C) % 16 != 0 || (ldc * esize) % 16 != 0) return GEMM_ERR_MISALIGNED;
    if (K > 0) {
        if (!A || !B || lda < K || ldb < K) return GEMM_ERR_INVALID_VALUE;
        if (reinterpret_cast<uintptr_t>(A) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0 || lda % 8 != 0 ||
            ldb % 8 != 0)
            return GEMM_ERR_MISALIGNED;
    }

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    DeviceState *ds = nullptr;
    st = device_state(device, &ds);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (K == 0) return launch_fill_zero(M, N, C, ldc, esize, ds->desc.num_sms, s);

    gemm_plan_t plan;
    st = make_plan(M, N, K, layout_a, layout_b, out_dtype, split_k, 1, ds->desc, main_kernel_desc(ds->regs_per_thread),
                   &plan);
    if (st != GEMM_OK) return st;
    const int64_t ldp = (N + 3) / 4 * 4;
    float *scratch = nullptr;
    if (plan.split_k > 1) {
        const int64_t per_split = M * ldp;   // < 2^62: M, N < 2^31
        if (per_split > static_cast<int64_t>(GEMM_NOALLOC_SCRATCH_FLOATS) ||
            plan.split_k > static_cast<int64_t>(GEMM_NOALLOC_SCRATCH_FLOATS) / per_split)
            return GEMM_ERR_INVALID_VALUE;
        st = noalloc_scratch(device, &scratch);
        if (st != GEMM_OK) return st;
    }

    CUtensorMap tmap_a, tmap_b;
    st = encode_operand(&tmap_a, A, K, M, lda, TILE_M);
    if (st != GEMM_OK) return st;
    st = encode_operand(&tmap_b, B, K, N, ldb, TILE_N);
    if (st != GEMM_OK) return st;

    KernelParams p{};
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((M + TILE_M - 1) / TILE_M);
    p.tiles_n = static_cast<int>((N + TILE_N - 1) / TILE_N);
    p.k_tiles = plan.k_tiles;
    p.split_k = plan.split_k;
    p.group_m = DEFAULT_RASTER_GROUP_M;
    p.num_units = plan.grid;
    if (plan.split_k > 1) {
        p.out = scratch;
        p.ld_out = ldp;
        p.split_stride = M * ldp;
        p.out_bf16 = 0;
    } else {
        p.out = C;
        p.ld_out = ldc;
        p.split_stride = 0;
        p.out_bf16 = out_dtype == GEMM_OUT_BF16 ? 1 : 0;
    }
    p.timeout_ns = static_cast<unsigned long long>(DEFAULT_TIMEOUT_MS) * 1000000ull;
    p.skip_load = 0;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.launch_ctas));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    if (cudaLaunchKernelEx(&cfg, gemm_bf16_tcgen05_kernel, tmap_a, tmap_b, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (plan.split_k > 1) {
        const long long total = M * ((N + 3) / 4);
        long long blocks = (total + 255) / 256;
        const long long cap = 4LL * ds->desc.num_sms;
        if (blocks > cap) blocks = cap;
        cudaLaunchConfig_t cc{};
        cc.gridDim = dim3(static_cast<unsigned>(blocks));
        cc.blockDim = dim3(256);
        cc.stream = s;
        if (cudaLaunchKernelEx(&cc, splitk_combine_kernel, static_cast<const float *>(scratch),
                               static_cast<long long>(ldp), static_cast<long long>(M * ldp), plan.split_k,
                               static_cast<int>(M), static_cast<int>(N), C, static_cast<long long>(ldc),
                               out_dtype == GEMM_OUT_BF16 ? 1 : 0) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    }
    return GEMM_OK;
}
