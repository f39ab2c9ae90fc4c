// splitk_tune.cu -- choosing the split count for a shape.
//
// The pages sweep the number of splits for fixed shapes (1, 2, 4, 8 and 16
// splits of M=32 N=512 K=2048 and M=96 N=512 K=512: "Aligned shared rows for
// pipelined NAX on CUDA", section "Measurement protocol"; "Wider
// consecutive-weight NAX GEMM", section "Performance method") and report that
// the best count depends on the shape.  Two ways to pick it here:
//
//   splitk_choose_splits    the planner's cost model, no device work;
//   splitk_autotune_splits  measurement: each candidate timed on the caller's
//                           buffers with CUDA events, from a CUDA graph of
//                           `reps` calls.
//
// Candidates are 1, 2, 4, 8 and 16 splits.  For a candidate n the split
// length is ceil(K / n) rounded up to a multiple of 32 and the split count is
// then ceil(K / length), which the contract requires (it can be below n when K
// is short, as with K=160 and n=4: length 64, 3 splits).

#include <cuda_runtime.h>

#include <algorithm>

#include "splitk.h"
#include "splitk_internal.h"

namespace {

constexpr int kCandidates = 5;
constexpr int64_t kCandidate[kCandidates] = {1, 2, 4, 8, 16};

void legal_split(int64_t K, int64_t n, int64_t *S, int64_t *kps)
{
    int64_t len = (K + n - 1) / n;
    len = (len + 31) / 32 * 32;
    *kps = len;
    *S = (K + len - 1) / len;
}

bool shape_ok(int64_t M, int64_t N, int64_t K)
{
    return M > 0 && M % 32 == 0 && N > 0 && N % 64 == 0 && K > 0 && K % 32 == 0 && M <= SPLITK_MAX_DIM &&
           N <= SPLITK_MAX_DIM && K <= SPLITK_MAX_DIM;
}

int elem_size(int dtype)
{
    switch (dtype) {
    case SPLITK_F32: return 4;
    case SPLITK_F16: case SPLITK_BF16: return 2;
    default: return 0;
    }
}

// Estimated microseconds per gemm_bt call in a graph of such calls: the
// tensor-core launch, plus for the two-kernel path (fused == 0, or a fused
// call that runs the two kernels) the reduce: 0.90 us, its bytes at ~3.2 TB/s
// and 0.047 us per split (fitted with the launch model in splitk_tc.cu).
double estimate_us(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, int dtype, int fused)
{
    const bool in_kernel = fused != 0 && splitk::fused_in_kernel(M, N, K, S, kps, dtype, false);
    const double reduce = 0.9016 + static_cast<double>(S + 1) * M * N * 4 / 3.192e6 + 0.0473 * static_cast<double>(S);
    return splitk::estimate_tc_us(M, N, K, S, kps, in_kernel, dtype == SPLITK_F32) + (in_kernel ? 0.0 : reduce);
}

}  // namespace

extern "C" {

int splitk_choose_splits(int64_t M, int64_t N, int64_t K, int dtype, int fused, int64_t *splits,
                         int64_t *k_per_split, double *model_us)
{
    if (!shape_ok(M, N, K)) return SPLITK_ERR_SHAPE;
    if (elem_size(dtype) == 0) return SPLITK_ERR_DTYPE;
    if (fused != 0 && fused != 1 && fused != 3) return SPLITK_ERR_CONFIG;
    if (!splits || !k_per_split) return SPLITK_ERR_NULL;
    double best = 1e300;
    int64_t bs = 0, bk = 0;
    for (int i = 0; i < kCandidates; ++i) {
        int64_t S, kps;
        legal_split(K, kCandidate[i], &S, &kps);
        if (model_us) model_us[i] = -1.0;
        if (splitk_check_geometry(M, N, K, S, kps) != SPLITK_OK) continue;
        const double t = estimate_us(M, N, K, S, kps, dtype, fused);
        if (model_us) model_us[i] = t;
        // candidates within 2% count as ties, won by the larger split count
        // (the measured curves are flat there, and more splits cost least
        // where the model misses a fixed cost)
        if (t <= best * 1.02) {
            best = std::min(best, t);
            bs = S;
            bk = kps;
        }
    }
    if (bs == 0) return SPLITK_ERR_SPLIT;
    *splits = bs;
    *k_per_split = bk;
    return SPLITK_OK;
}

int splitk_autotune_splits(const void *A, const void *B, float *out, void *workspace, size_t workspace_bytes,
                           int64_t M, int64_t N, int64_t K, int dtype, int fused, int reps, void *stream,
                           int64_t *splits, int64_t *k_per_split, float *us)
{
    if (!shape_ok(M, N, K)) return SPLITK_ERR_SHAPE;
    if (elem_size(dtype) == 0) return SPLITK_ERR_DTYPE;
    if ((fused != 0 && fused != 1 && fused != 3) || reps < 1 || reps > 1000) return SPLITK_ERR_CONFIG;
    if (!splits || !k_per_split) return SPLITK_ERR_NULL;
    // every candidate's arguments are checked before anything is enqueued
    int64_t cs[kCandidates], ck[kCandidates];
    bool run[kCandidates];
    int runnable = 0, first_error = SPLITK_OK;
    for (int i = 0; i < kCandidates; ++i) {
        legal_split(K, kCandidate[i], &cs[i], &ck[i]);
        const int st = splitk::check_gemm_bt(A, B, out, workspace, workspace_bytes, M, N, K, cs[i], ck[i], dtype,
                                             fused);
        bool dup = false;
        for (int j = 0; j < i; ++j) dup = dup || (run[j] && cs[j] == cs[i]);
        run[i] = st == SPLITK_OK && !dup;
        if (st != SPLITK_OK && st != SPLITK_ERR_WORKSPACE && first_error == SPLITK_OK) first_error = st;
        runnable += run[i] ? 1 : 0;
        if (us) us[i] = -1.0f;
    }
    if (first_error != SPLITK_OK) return first_error;
    if (runnable == 0) return SPLITK_ERR_WORKSPACE;   // not even one split fits the workspace

    cudaStream_t user = static_cast<cudaStream_t>(stream), ts = nullptr;
    cudaEvent_t ready = nullptr, e0 = nullptr, e1 = nullptr;
    int rc = SPLITK_OK;
    auto cuda = [&](cudaError_t e, const char *what) {
        if (e != cudaSuccess && rc == SPLITK_OK) {
            splitk::note_error(e, what);
            rc = SPLITK_ERR_CUDA;
        }
        return e == cudaSuccess;
    };
    // timing runs on a private stream, after the work already on `stream`
    if (!cuda(cudaStreamCreateWithFlags(&ts, cudaStreamNonBlocking), "cudaStreamCreate") ||
        !cuda(cudaEventCreate(&ready), "cudaEventCreate") || !cuda(cudaEventCreate(&e0), "cudaEventCreate") ||
        !cuda(cudaEventCreate(&e1), "cudaEventCreate") || !cuda(cudaEventRecord(ready, user), "cudaEventRecord") ||
        !cuda(cudaStreamWaitEvent(ts, ready, 0), "cudaStreamWaitEvent")) {
        // fall through to clean-up
    }
    float best = 3.0e38f;
    int bi = -1;
    for (int i = 0; i < kCandidates && rc == SPLITK_OK; ++i) {
        if (!run[i]) continue;
        const int w = gemm_bt(A, B, out, workspace, workspace_bytes, M, N, K, cs[i], ck[i], dtype, fused, ts);
        if (w != SPLITK_OK) {
            rc = w;
            break;
        }
        cudaGraph_t g = nullptr;
        cudaGraphExec_t ge = nullptr;
        if (!cuda(cudaStreamBeginCapture(ts, cudaStreamCaptureModeThreadLocal), "cudaStreamBeginCapture")) break;
        int cap = SPLITK_OK;
        for (int r = 0; r < reps && cap == SPLITK_OK; ++r)
            cap = gemm_bt(A, B, out, workspace, workspace_bytes, M, N, K, cs[i], ck[i], dtype, fused, ts);
        const bool ended = cuda(cudaStreamEndCapture(ts, &g), "cudaStreamEndCapture");
        if (cap != SPLITK_OK && rc == SPLITK_OK) rc = cap;
        if (ended && rc == SPLITK_OK && cuda(cudaGraphInstantiate(&ge, g, 0), "cudaGraphInstantiate")) {
            constexpr int kRounds = 3;
            cuda(cudaGraphLaunch(ge, ts), "cudaGraphLaunch");   // warm
            cuda(cudaEventRecord(e0, ts), "cudaEventRecord");
            for (int r = 0; r < kRounds; ++r) cuda(cudaGraphLaunch(ge, ts), "cudaGraphLaunch");
            cuda(cudaEventRecord(e1, ts), "cudaEventRecord");
            float ms = 0.f;
            if (cuda(cudaEventSynchronize(e1), "cudaEventSynchronize") &&
                cuda(cudaEventElapsedTime(&ms, e0, e1), "cudaEventElapsedTime")) {
                const float t = ms * 1000.0f / static_cast<float>(kRounds * reps);
                if (us) us[i] = t;
                if (t < best) {
                    best = t;
                    bi = i;
                }
            }
        }
        if (ge) cudaGraphExecDestroy(ge);
        if (g) cudaGraphDestroy(g);
        if (rc == SPLITK_OK && splitk_get_device_status(ts) != SPLITK_OK) rc = SPLITK_ERR_DEVICE_TIMEOUT;
    }
    if (rc == SPLITK_OK && bi >= 0) {
        // leave `out` holding the chosen split's result
        const int w = gemm_bt(A, B, out, workspace, workspace_bytes, M, N, K, cs[bi], ck[bi], dtype, fused, ts);
        if (w != SPLITK_OK) rc = w;
        cuda(cudaEventRecord(e1, ts), "cudaEventRecord");
        cuda(cudaStreamWaitEvent(user, e1, 0), "cudaStreamWaitEvent");   // `stream` sees the final call
        cuda(cudaStreamSynchronize(ts), "cudaStreamSynchronize");
        *splits = cs[bi];
        *k_per_split = ck[bi];
    }
    if (ts) cudaStreamSynchronize(ts);
    if (ready) cudaEventDestroy(ready);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (ts) cudaStreamDestroy(ts);
    if (rc == SPLITK_OK && bi < 0) rc = SPLITK_ERR_CUDA;
    return rc;
}

}  // extern "C"
