// Compile-time shape of the main GEMM kernel, shared by the planner and the
// CUDA sources.  One CTA computes a TILE_M x TILE_N block of C; operands
// arrive in TILE_K-wide k-tiles through a STAGES-deep shared-memory ring.
#pragma once

namespace gemm {

constexpr int TILE_M = 128;              // rows of C per CTA (= MMA M, one TMEM lane per row)
constexpr int TILE_N = 256;              // columns of C per CTA (= MMA N)
constexpr int TILE_K = 64;               // bf16 elements per k-tile row: 128 bytes, one swizzle span
constexpr int MMA_K = 16;                // K of one kind::f16 tcgen05.mma
constexpr int STAGES = 4;                // operand ring depth
constexpr int ACC_BUFS = 2;              // accumulators in TMEM (epilogue overlaps the next tile)
constexpr int TMEM_COLS = ACC_BUFS * TILE_N;   // fp32 accumulator: one column per element of a row

constexpr int NUM_WARPS = 6;             // 0: TMA producer, 1: MMA issuer, 2..5: epilogue
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int EPI_THREADS = 128;

constexpr int A_STAGE_BYTES = TILE_M * TILE_K * 2;
constexpr int B_STAGE_BYTES = TILE_N * TILE_K * 2;
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int NUM_BARRIERS = 2 * STAGES + 2 * ACC_BUFS + 1;
// ring + barriers + TMEM address slot + abort flag, plus 1 KiB to align the
// ring to the 1024-byte swizzle atom
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARRIERS * 8 + 16;

constexpr int DEFAULT_RASTER_GROUP_M = 16;
constexpr int DEFAULT_TIMEOUT_MS = 4000;
constexpr int MIN_K_TILES_PER_SPLIT = 4;  // automatic split-K keeps at least this many k-tiles per slice

}  // namespace gemm
