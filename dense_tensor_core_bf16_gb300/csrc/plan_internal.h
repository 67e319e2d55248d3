// Planner internals shared by plan.cpp and the CUDA launcher.
#pragma once
#include "gemm_bf16.h"

namespace gemm {

gemm_status_t check_problem(int64_t M, int64_t N, int64_t K, gemm_layout_t la, gemm_layout_t lb,
                            gemm_dtype_t out, int split_k);
gemm_status_t occupancy(const gemm_kernel_desc_t &k, const gemm_device_desc_t &d, int *b, int *limiter);
// allow_stream_k: false for callers without a growable workspace.
gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, gemm_layout_t la, gemm_layout_t lb,
                        gemm_dtype_t out, const gemm_options_t &o, bool allow_stream_k,
                        const gemm_device_desc_t &dev, const gemm_kernel_desc_t &kern, gemm_plan_t *plan);
int resolve_variant(int requested);
int choose_variant(int64_t M, int64_t N, int64_t K, int requested, int split_k, const gemm_device_desc_t &dev);
int choose_split(int64_t tiles, int k_tiles, int capacity, int requested, int64_t K);
// First stream-K iteration of each cluster, bounds[0 .. clusters] (the last is
// sk_iters), for the tail a plan with these options runs.
void stream_k_bounds(int64_t sk_iters, int64_t clusters, int64_t k_tiles, const gemm_options_t &o, int64_t *bounds);
gemm_status_t conv_check(const gemm_conv2d_desc_t *d, int64_t *P, int64_t *Q);
// Frees the host-batch staging slots of every device (host_pipeline.cpp).
void release_host_staging();

}  // namespace gemm
