// Host-resident GEMMs (gemm_bf16_host_batch in gemm_bf16.h): operands copied
// into device staging slots, products by gemm_bf16_ex, results copied back,
// with the copies of one problem overlapped with the product of another.
//
// Per device: two staging slots (A, B, C buffers each), kLanes operand-copy
// streams, one product stream and one result-copy stream, all created
// non-blocking.  Problem i takes slot i mod 2 (counted across calls).  The
// order on the device is kept by events alone:
//   operand lanes:  wait slot.comp_done (its A, B no longer read), and with a
//                   C input also slot.out_done; copy; record slot.in_done[j]
//   product stream: wait every slot.in_done[j] and slot.out_done (its C no
//                   longer being copied out); gemm_bf16_ex; record comp_done
//   result stream:  wait slot.comp_done; copy C out; record slot.out_done
// so while problem i's product runs, problem i+1's operands fill the other
// slot and problem i-1's result drains from it.  Each operand is split by rows
// over the lanes so that several copy engines share the transfer.
#include "gemm_bf16.h"
#include "plan_internal.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace gemm {
namespace {

constexpr int kSlots = 2;
constexpr int kLanes = 2;
constexpr int kMaxPipes = 64;

struct Slot {
    void *a = nullptr, *b = nullptr, *c = nullptr;
    size_t a_bytes = 0, b_bytes = 0, c_bytes = 0;
    cudaEvent_t in_done[kLanes] = {};
    cudaEvent_t comp_done = nullptr, out_done = nullptr;
};

struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t lane[kLanes] = {};
    cudaStream_t comp = nullptr, out = nullptr;
    cudaEvent_t start = nullptr;
    Slot slot[kSlots];
    uint64_t next = 0;
};

HostPipe g_pipes[kMaxPipes];

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// One matrix as the copies see it: `rows` rows of `width` elements.
struct Extent {
    int64_t rows, width, host_ld, dev_ld;
    int esize;
    size_t dev_bytes() const { return static_cast<size_t>(rows * dev_ld * esize); }
};

// Device rows are padded to 16 bytes, the TMA stride rule.
Extent extent(int64_t rows, int64_t width, int64_t host_ld, int esize) {
    return Extent{rows, width, host_ld, round_up(width > 0 ? width : 1, 16 / esize), esize};
}

Extent extent_a(const gemm_host_problem_t &p) {
    return p.layout_a == GEMM_ROW_MAJOR ? extent(p.M, p.K, p.lda, 2) : extent(p.K, p.M, p.lda, 2);
}
Extent extent_b(const gemm_host_problem_t &p) {
    return p.layout_b == GEMM_COL_MAJOR ? extent(p.N, p.K, p.ldb, 2) : extent(p.K, p.N, p.ldb, 2);
}
Extent extent_c(const gemm_host_problem_t &p, gemm_dtype_t out) {
    return extent(p.M, p.N, p.ldc, out == GEMM_OUT_BF16 ? 2 : 4);
}

bool ok(cudaError_t e) {
    if (e == cudaSuccess) return true;
    cudaGetLastError();
    return false;
}

// Rows [r0, r1) of a matrix between host and device.
bool copy_rows(const Extent &e, void *dev, const void *host, int64_t r0, int64_t r1, bool to_device,
               cudaStream_t s) {
    if (r1 <= r0 || e.width == 0) return true;
    const size_t hp = static_cast<size_t>(e.host_ld * e.esize), dp = static_cast<size_t>(e.dev_ld * e.esize);
    const size_t w = static_cast<size_t>(e.width * e.esize);
    char *d = static_cast<char *>(dev) + static_cast<size_t>(r0) * dp;
    // cudaMemcpyDefault: the direction follows from the addresses (unified
    // addressing), so a device pointer passed as a "host" array still works.
    if (to_device) {
        const char *h = static_cast<const char *>(host) + static_cast<size_t>(r0) * hp;
        return ok(cudaMemcpy2DAsync(d, dp, h, hp, w, static_cast<size_t>(r1 - r0), cudaMemcpyDefault, s));
    }
    char *h = static_cast<char *>(const_cast<void *>(host)) + static_cast<size_t>(r0) * hp;
    return ok(cudaMemcpy2DAsync(h, hp, d, dp, w, static_cast<size_t>(r1 - r0), cudaMemcpyDefault, s));
}

gemm_status_t create_pipe(HostPipe &p) {
    if (p.ready) return GEMM_OK;
    bool good = true;
    for (int j = 0; j < kLanes; ++j) good = good && ok(cudaStreamCreateWithFlags(&p.lane[j], cudaStreamNonBlocking));
    good = good && ok(cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking));
    good = good && ok(cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking));
    good = good && ok(cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming));
    for (Slot &s : p.slot) {
        for (int j = 0; j < kLanes; ++j) good = good && ok(cudaEventCreateWithFlags(&s.in_done[j], cudaEventDisableTiming));
        good = good && ok(cudaEventCreateWithFlags(&s.comp_done, cudaEventDisableTiming));
        good = good && ok(cudaEventCreateWithFlags(&s.out_done, cudaEventDisableTiming));
    }
    if (!good) return GEMM_ERR_LAUNCH;
    p.ready = true;
    return GEMM_OK;
}

void sync_pipe(HostPipe &p) {
    for (int j = 0; j < kLanes; ++j) cudaStreamSynchronize(p.lane[j]);
    cudaStreamSynchronize(p.comp);
    cudaStreamSynchronize(p.out);
    cudaGetLastError();
}

void free_slots(HostPipe &p) {
    for (Slot &s : p.slot) {
        cudaFree(s.a);
        cudaFree(s.b);
        cudaFree(s.c);
        s.a = s.b = s.c = nullptr;
        s.a_bytes = s.b_bytes = s.c_bytes = 0;
    }
    cudaGetLastError();
}

// Every slot holds at least the given bytes; growing waits for the pipe first.
gemm_status_t ensure_slots(HostPipe &p, size_t a, size_t b, size_t c) {
    const Slot &s0 = p.slot[0];
    if (s0.a_bytes >= a && s0.b_bytes >= b && s0.c_bytes >= c) return GEMM_OK;
    sync_pipe(p);
    const size_t na = a > s0.a_bytes ? a : s0.a_bytes, nb = b > s0.b_bytes ? b : s0.b_bytes,
                 nc = c > s0.c_bytes ? c : s0.c_bytes;
    free_slots(p);
    for (Slot &s : p.slot) {
        if ((na && !ok(cudaMalloc(&s.a, na))) || (nb && !ok(cudaMalloc(&s.b, nb))) || (nc && !ok(cudaMalloc(&s.c, nc)))) {
            free_slots(p);
            return GEMM_ERR_OUT_OF_MEMORY;
        }
        s.a_bytes = na;
        s.b_bytes = nb;
        s.c_bytes = nc;
    }
    return GEMM_OK;
}

// The host-side checks first (no CUDA call), then the plan on the current
// device, which also rejects what the library cannot run.
gemm_status_t check_host_problem(const gemm_host_problem_t &p, gemm_dtype_t out, const gemm_options_t *opts) {
    gemm_status_t st = check_problem(p.M, p.N, p.K, p.layout_a, p.layout_b, out, opts ? opts->split_k : 0);
    if (st != GEMM_OK) return st;
    if (p.M == 0 || p.N == 0) return GEMM_OK;
    if (!p.C || p.ldc < p.N) return GEMM_ERR_INVALID_VALUE;
    if (p.K > 0) {
        const int64_t min_lda = p.layout_a == GEMM_ROW_MAJOR ? p.K : p.M;
        const int64_t min_ldb = p.layout_b == GEMM_COL_MAJOR ? p.K : p.N;
        if (!p.A || !p.B || p.lda < min_lda || p.ldb < min_ldb) return GEMM_ERR_INVALID_VALUE;
    }
    return GEMM_OK;
}

gemm_status_t check_options(const gemm_options_t *opts) {
    if (!opts) return GEMM_OK;
    const gemm_options_t &o = *opts;
    if (o.timeout_ms < 0 || o.raster_group_m < 0 || o.debug_skip_load < 0 || o.split_k < 0) return GEMM_ERR_INVALID_VALUE;
    if (o.epilogue) {
        if (o.epilogue->activation < GEMM_ACT_NONE || o.epilogue->activation > GEMM_ACT_GELU)
            return GEMM_ERR_INVALID_VALUE;
        if (reinterpret_cast<uintptr_t>(o.epilogue->bias) % 16 != 0) return GEMM_ERR_MISALIGNED;
    }
    return GEMM_OK;
}

// Rows of a matrix dealt to lane j of kLanes, in order.
void lane_rows(int64_t rows, int j, int64_t *r0, int64_t *r1) {
    *r0 = rows * j / kLanes;
    *r1 = rows * (j + 1) / kLanes;
}

}  // namespace

void release_host_staging() {
    int current = -1;
    if (!ok(cudaGetDevice(&current))) return;
    for (int d = 0; d < kMaxPipes; ++d) {
        HostPipe &p = g_pipes[d];
        std::lock_guard<std::mutex> lock(p.mu);
        if (!p.ready) continue;
        if (!ok(cudaSetDevice(d))) continue;
        sync_pipe(p);
        free_slots(p);
    }
    cudaSetDevice(current);
    cudaGetLastError();
}

}  // namespace gemm

using namespace gemm;

extern "C" gemm_status_t gemm_bf16_host_batch(int64_t count, const gemm_host_problem_t *problems,
                                              gemm_dtype_t out_dtype, const gemm_options_t *opts, void *stream) {
    if (count < 0 || (count > 0 && !problems)) return GEMM_ERR_INVALID_VALUE;
    gemm_status_t st = check_options(opts);
    if (st != GEMM_OK) return st;
    if (out_dtype != GEMM_OUT_F32 && out_dtype != GEMM_OUT_BF16) return GEMM_ERR_INVALID_VALUE;
    const bool c_in = opts && opts->epilogue && opts->epilogue->beta != 0.0f;
    if (count == 0) return GEMM_OK;
    size_t need_a = 0, need_b = 0, need_c = 0;
    for (int64_t i = 0; i < count; ++i) {
        st = check_host_problem(problems[i], out_dtype, opts);
        if (st != GEMM_OK) return st;
    }
    for (int64_t i = 0; i < count; ++i) {
        const gemm_host_problem_t &p = problems[i];
        if (p.M == 0 || p.N == 0) continue;
        if (p.K > 0) {
            gemm_plan_t plan;
            st = gemm_plan(p.M, p.N, p.K, p.layout_a, p.layout_b, out_dtype, opts, &plan);
            if (st != GEMM_OK) return st;
        }
        const size_t a = p.K > 0 ? extent_a(p).dev_bytes() : 0, b = p.K > 0 ? extent_b(p).dev_bytes() : 0;
        const size_t c = extent_c(p, out_dtype).dev_bytes();
        need_a = a > need_a ? a : need_a;
        need_b = b > need_b ? b : need_b;
        need_c = c > need_c ? c : need_c;
    }
    if (need_c == 0) return GEMM_OK;   // every problem empty

    int device = 0;
    if (!ok(cudaGetDevice(&device))) return GEMM_ERR_NO_DEVICE;
    if (device < 0 || device >= kMaxPipes) return GEMM_ERR_NO_DEVICE;
    HostPipe &pipe = g_pipes[device];
    std::lock_guard<std::mutex> lock(pipe.mu);
    st = create_pipe(pipe);
    if (st != GEMM_OK) return st;
    st = ensure_slots(pipe, need_a, need_b, need_c);
    if (st != GEMM_OK) return st;

    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    if (!ok(cudaEventRecord(pipe.start, caller))) return GEMM_ERR_LAUNCH;
    bool good = true;
    for (int j = 0; j < kLanes; ++j) good = good && ok(cudaStreamWaitEvent(pipe.lane[j], pipe.start, 0));
    good = good && ok(cudaStreamWaitEvent(pipe.comp, pipe.start, 0));
    good = good && ok(cudaStreamWaitEvent(pipe.out, pipe.start, 0));
    const Slot *last = nullptr;
    for (int64_t i = 0; good && i < count; ++i) {
        const gemm_host_problem_t &p = problems[i];
        if (p.M == 0 || p.N == 0) continue;
        Slot &sl = pipe.slot[pipe.next++ % kSlots];
        const Extent ea = extent_a(p), eb = extent_b(p), ec = extent_c(p, out_dtype);
        for (int j = 0; good && j < kLanes; ++j) {
            cudaStream_t ls = pipe.lane[j];
            good = ok(cudaStreamWaitEvent(ls, sl.comp_done, 0));
            int64_t r0, r1;
            if (good && c_in) {
                good = ok(cudaStreamWaitEvent(ls, sl.out_done, 0));
                lane_rows(ec.rows, j, &r0, &r1);
                good = good && copy_rows(ec, sl.c, p.C, r0, r1, true, ls);
            }
            if (good && p.K > 0) {
                lane_rows(ea.rows, j, &r0, &r1);
                good = copy_rows(ea, sl.a, p.A, r0, r1, true, ls);
                lane_rows(eb.rows, j, &r0, &r1);
                good = good && copy_rows(eb, sl.b, p.B, r0, r1, true, ls);
            }
            good = good && ok(cudaEventRecord(sl.in_done[j], ls));
        }
        for (int j = 0; good && j < kLanes; ++j) good = ok(cudaStreamWaitEvent(pipe.comp, sl.in_done[j], 0));
        good = good && ok(cudaStreamWaitEvent(pipe.comp, sl.out_done, 0));
        if (!good) break;
        st = gemm_bf16_ex(p.M, p.N, p.K, sl.a, ea.dev_ld, sl.b, eb.dev_ld, sl.c, ec.dev_ld, p.layout_a, p.layout_b,
                          out_dtype, opts, pipe.comp);
        if (st != GEMM_OK) break;
        good = ok(cudaEventRecord(sl.comp_done, pipe.comp));
        good = good && ok(cudaStreamWaitEvent(pipe.out, sl.comp_done, 0));
        good = good && copy_rows(ec, sl.c, p.C, 0, ec.rows, false, pipe.out);
        good = good && ok(cudaEventRecord(sl.out_done, pipe.out));
        last = &sl;
    }
    // Even after a failure the caller's stream waits for what was enqueued,
    // so that the host arrays it covers are not released under the copies.
    if (last && !ok(cudaStreamWaitEvent(caller, last->out_done, 0))) return GEMM_ERR_LAUNCH;
    if (st != GEMM_OK || !good) {
        // A problem that failed before its result copy may still have operand
        // copies (and part of its product) in flight: wait for every lane and
        // the product stream too.  `start` is free to record again: each wait
        // takes the event as last recorded when the wait is enqueued.
        for (int j = 0; j < kLanes; ++j)
            if (ok(cudaEventRecord(pipe.start, pipe.lane[j]))) ok(cudaStreamWaitEvent(caller, pipe.start, 0));
        if (ok(cudaEventRecord(pipe.start, pipe.comp))) ok(cudaStreamWaitEvent(caller, pipe.start, 0));
    }
    if (st != GEMM_OK) return st;
    return good ? GEMM_OK : GEMM_ERR_LAUNCH;
}
