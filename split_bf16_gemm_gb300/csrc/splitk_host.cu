// splitk_host.cu -- gemm_bt for activations and results in host memory.
//
// The pages time the operation on operands already resident on the device
// (weights prepared and uploaded once, outside timing: "Wider
// consecutive-weight NAX GEMM", section "Performance method").  A serving
// loop also has to bring each batch of activations in and each result out.
// This entry point does that for `count` operations as a three-stage
// pipeline on the current device:
//
//   copy-in stream   A_host[g] -> staging A slots         (group g)
//   caller's stream  the operations of group g (after its copy-in): one
//                    launch for fused calls whose plan groups, else gemm_bt
//                    on each
//   copy-out stream  staging out slots -> out_host[g]     (after its compute)
//
// A group is `ops_per_copy` consecutive operations moved by one copy each way,
// so the copy-in of group g+1 and the copy-out of group g-1 run on the copy
// engines while group g computes.  Events order the stages; the caller's
// stream waits for the last copy-out before the call's work counts as done on
// it.  The copy-in waits only for the previous call on the same staging (an
// event the library keeps per staging buffer), or, the first time a staging
// is seen, for everything the caller's stream held before the call.  A
// caller alternating two staging buffers therefore gets the next batch's
// activations in while the current batch computes.
//
// The two copy streams and four events per device are created on the first
// call on that device and kept until the process exits.  One mutex per
// process serialises the enqueueing of concurrent calls (the events are
// shared); their device work still runs in stream order.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "splitk.h"
#include "splitk_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxCount = 1 << 16;
constexpr size_t kSlotAlign = 256;

struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, loaded = nullptr, computed = nullptr, drained = nullptr;
};

// The end of the last call on each staging buffer (most recent first).
constexpr int kTracked = 32;
struct LastUse {
    int device = -1;
    const void *staging = nullptr;
    cudaEvent_t done = nullptr;
    uint64_t stamp = 0;
};

std::mutex g_mu;
Pipe g_pipes[kMaxDevices];
LastUse g_last[kTracked];
uint64_t g_clock = 0;

// The entry for (device, staging): found, or the least recently used slot
// taken over (its event kept, its staging replaced).  *known says whether the
// staging had an entry.
LastUse *last_use(int device, const void *staging, bool *known)
{
    LastUse *lru = &g_last[0];
    for (LastUse &e : g_last) {
        if (e.device == device && e.staging == staging) {
            *known = true;
            e.stamp = ++g_clock;
            return &e;
        }
        if (e.stamp < lru->stamp) lru = &e;
    }
    *known = false;
    if (lru->done && lru->device != device) {   // an event belongs to its device
        cudaEventDestroy(lru->done);
        lru->done = nullptr;
    }
    lru->device = device;
    lru->staging = staging;
    lru->stamp = ++g_clock;
    return lru;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elem_size(int dtype)
{
    switch (dtype) {
    case SPLITK_F32: return 4;
    case SPLITK_F16: case SPLITK_BF16: return 2;
    default: return 0;
    }
}

struct Layout {
    size_t a_bytes, out_bytes;     // one operation's slot of each
    size_t a_off, out_off, ws_off; // offsets into the staging
    size_t ws_bytes, total;
};

// Staging: count A slots, then count out slots, then one gemm_bt workspace.
// A and out slots are packed back to back (M*K*elem and M*N*4 are multiples
// of 2048 bytes under the contract), so a group is one contiguous range.
Layout layout_for(int64_t count, int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, int e)
{
    Layout L{};
    L.a_bytes = static_cast<size_t>(M * K) * e;
    L.out_bytes = static_cast<size_t>(M * N) * 4;
    L.a_off = 0;
    L.out_off = round_up(L.a_bytes * count, kSlotAlign);
    L.ws_off = round_up(L.out_off + L.out_bytes * count, kSlotAlign);
    L.ws_bytes = gemm_bt_workspace_bytes(M, N, K, S, kps, 1);
    L.total = L.ws_off + L.ws_bytes;
    return L;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fail(cudaError_t e, const char *what)
{
    splitk::note_error(e, what);
    return SPLITK_ERR_CUDA;
}

int pipe_for_current_device(Pipe **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        splitk::note_message("gemm_bt_host_batch: device index beyond the supported range", dev);
        return SPLITK_ERR_CUDA;
    }
    Pipe &p = g_pipes[dev];
    if (!p.ready) {
        if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.loaded, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.computed, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.drained, cudaEventDisableTiming)) != cudaSuccess)
            return fail(e, "creating the host pipeline's streams and events");
        p.ready = true;
    }
    *out = &p;
    return SPLITK_OK;
}

// Operations per copy when the caller leaves it to the library: enough that
// one copy moves at least 4 MiB of A (a pinned copy reaches about 140 GB/s at
// 1 MiB, 170 at 2 MiB and 200 at 8 MiB on GB300, and the operations of a
// group run as one launch where they can), but at most half the batch, so
// that copies still overlap compute.  Batches of eight BF16 M256 N1024
// K2048 operations on GB300, two streams alternated: 9.1 us per operation
// with two per copy, 8.1 with four, 8.7 with eight.
int64_t auto_ops_per_copy(int64_t count, size_t a_bytes)
{
    const size_t target = size_t(4) << 20;
    int64_t g = static_cast<int64_t>((target + a_bytes - 1) / a_bytes);
    const int64_t half = (count + 1) / 2;
    if (g > half) g = half;
    return g < 1 ? 1 : g;
}

}  // namespace

extern "C" {

size_t gemm_bt_host_staging_bytes(int64_t count, int64_t M, int64_t N, int64_t K, int64_t splits,
                                  int64_t k_per_split, int dtype)
{
    if (count <= 0 || count > kMaxCount) return 0;
    const int e = elem_size(dtype);
    if (e == 0 || splitk_check_geometry(M, N, K, splits, k_per_split) != SPLITK_OK) return 0;
    return layout_for(count, M, N, K, splits, k_per_split, e).total;
}

int gemm_bt_host_batch(const void *A_host, const void *const *B, float *out_host, int64_t count, void *staging,
                       size_t staging_bytes, int64_t M, int64_t N, int64_t K, int64_t splits, int64_t k_per_split,
                       int dtype, int fused, int64_t ops_per_copy, void *stream)
{
    // --- validation: nothing is enqueued unless all of it passes
    const int geo = splitk_check_geometry(M, N, K, splits, k_per_split);
    if (geo != SPLITK_OK) return geo;
    const int e = elem_size(dtype);
    if (e == 0) return SPLITK_ERR_DTYPE;
    if (count <= 0 || count > kMaxCount || ops_per_copy < 0) return SPLITK_ERR_CONFIG;
    if (fused != 0 && fused != 1 && fused != 3) return SPLITK_ERR_CONFIG;
    if (!A_host || !B || !out_host || !staging) return SPLITK_ERR_NULL;
    if (!aligned16(staging)) return SPLITK_ERR_ALIGN;
    const Layout L = layout_for(count, M, N, K, splits, k_per_split, e);
    if (staging_bytes < L.total) return SPLITK_ERR_WORKSPACE;
    const size_t b_bytes = static_cast<size_t>(N * K) * e;
    for (int64_t i = 0; i < count; ++i) {
        if (!B[i]) return SPLITK_ERR_NULL;
        if (!aligned16(B[i])) return SPLITK_ERR_ALIGN;
        if (overlap(B[i], b_bytes, staging, L.total)) return SPLITK_ERR_ALIAS;
    }
    if (overlap(A_host, L.a_bytes * count, out_host, L.out_bytes * count)) return SPLITK_ERR_ALIAS;
    if (overlap(A_host, L.a_bytes * count, staging, L.total) || overlap(out_host, L.out_bytes * count, staging, L.total))
        return SPLITK_ERR_ALIAS;

    const int64_t g = ops_per_copy > 0 ? (ops_per_copy < count ? ops_per_copy : count)
                                       : auto_ops_per_copy(count, L.a_bytes);
    char *const st = static_cast<char *>(staging);
    char *const a_dev = st + L.a_off;
    float *const out_dev = reinterpret_cast<float *>(st + L.out_off);
    void *const ws = st + L.ws_off;
    const char *const a_src = static_cast<const char *>(A_host);
    char *const o_dst = reinterpret_cast<char *>(out_host);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // One launch per group where the calls are fused in the launch and their
    // plan allows it (the same sums as one call each).
    const bool batchable = fused == 1 && dtype != SPLITK_F32 &&
                           splitk::fused_in_kernel(M, N, K, splits, k_per_split, dtype, false) &&
                           splitk::batch_possible(M, N, K, splits, k_per_split);

    std::lock_guard<std::mutex> lock(g_mu);
    Pipe *p = nullptr;
    int rc = pipe_for_current_device(&p);
    if (rc != SPLITK_OK) return rc;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return fail(ce, "cudaGetDevice");
    bool known = false;
    LastUse *use = last_use(dev, staging, &known);
    if (!use->done && (ce = cudaEventCreateWithFlags(&use->done, cudaEventDisableTiming)) != cudaSuccess) {
        use->device = -1;
        return fail(ce, "cudaEventCreate(staging)");
    }

    // the copy-in overwrites the staging's A slots: after the previous call on
    // this staging, or, for a staging not seen before, after everything
    // already on the caller's stream (zeroing it, for one)
    if (known) {
        if ((ce = cudaStreamWaitEvent(p->in, use->done, 0)) != cudaSuccess)
            return fail(ce, "cudaStreamWaitEvent(staging)");
    } else {
        if ((ce = cudaEventRecord(p->start, s)) != cudaSuccess) return fail(ce, "cudaEventRecord(start)");
        if ((ce = cudaStreamWaitEvent(p->in, p->start, 0)) != cudaSuccess)
            return fail(ce, "cudaStreamWaitEvent(start)");
    }

    for (int64_t g0 = 0; g0 < count && rc == SPLITK_OK; g0 += g) {
        const int64_t n = (count - g0 < g) ? count - g0 : g;
        ce = cudaMemcpyAsync(a_dev + L.a_bytes * g0, a_src + L.a_bytes * g0, L.a_bytes * n, cudaMemcpyDefault, p->in);
        if (ce != cudaSuccess) { rc = fail(ce, "cudaMemcpyAsync(A in)"); break; }
        if ((ce = cudaEventRecord(p->loaded, p->in)) != cudaSuccess) { rc = fail(ce, "cudaEventRecord(loaded)"); break; }
        if ((ce = cudaStreamWaitEvent(s, p->loaded, 0)) != cudaSuccess) { rc = fail(ce, "cudaStreamWaitEvent(loaded)"); break; }
        for (int64_t i = g0; i < g0 + n && rc == SPLITK_OK;) {
            // fused calls whose splits are summed in the launch: up to
            // kMaxGroup of the group in one launch; else one call each
            // (a lone operation keeps gemm_bt's own plan, which spreads it
            // over more of the SMs)
            const int64_t b = batchable ? std::min<int64_t>(g0 + n - i, splitk::kMaxGroup) : 0;
            if (b > 1) {
                const void *as[splitk::kMaxGroup];
                float *os[splitk::kMaxGroup];
                for (int64_t j = 0; j < b; ++j) {
                    as[j] = a_dev + L.a_bytes * (i + j);
                    os[j] = out_dev + static_cast<size_t>(M * N) * (i + j);
                }
                rc = splitk::run_fused_batch(as, B + i, os, static_cast<int>(b), M, N, K, splits, k_per_split, dtype,
                                             s);
                i += b;
            } else {
                rc = gemm_bt(a_dev + L.a_bytes * i, B[i], out_dev + static_cast<size_t>(M * N) * i, ws, L.ws_bytes,
                             M, N, K, splits, k_per_split, dtype, fused, stream);
                ++i;
            }
        }
        if (rc != SPLITK_OK) break;
        if ((ce = cudaEventRecord(p->computed, s)) != cudaSuccess) { rc = fail(ce, "cudaEventRecord(computed)"); break; }
        if ((ce = cudaStreamWaitEvent(p->out, p->computed, 0)) != cudaSuccess) { rc = fail(ce, "cudaStreamWaitEvent(computed)"); break; }
        ce = cudaMemcpyAsync(o_dst + L.out_bytes * g0, reinterpret_cast<char *>(out_dev) + L.out_bytes * g0,
                             L.out_bytes * n, cudaMemcpyDefault, p->out);
        if (ce != cudaSuccess) { rc = fail(ce, "cudaMemcpyAsync(out)"); break; }
    }
    // join: the caller's stream holds the whole batch, copies included (also
    // after a failure part-way, so that what was enqueued stays ordered)
    const cudaError_t j1 = cudaEventRecord(p->drained, p->out);
    const cudaError_t j2 = j1 == cudaSuccess ? cudaStreamWaitEvent(s, p->drained, 0) : j1;
    const cudaError_t j3 = cudaEventRecord(p->drained, p->in);
    const cudaError_t j4 = j3 == cudaSuccess ? cudaStreamWaitEvent(s, p->drained, 0) : j3;
    if (rc == SPLITK_OK && j2 != cudaSuccess) return fail(j2, "joining the copy-out stream");
    if (rc == SPLITK_OK && j4 != cudaSuccess) return fail(j4, "joining the copy-in stream");
    // the end of this call's work on the staging, for the next call on it
    ce = cudaEventRecord(use->done, s);
    if (ce != cudaSuccess) {
        use->device = -1;   // forget the staging: the next call waits on the caller's stream
        if (rc == SPLITK_OK) return fail(ce, "cudaEventRecord(staging)");
    }
    return rc;
}

}  // extern "C"
