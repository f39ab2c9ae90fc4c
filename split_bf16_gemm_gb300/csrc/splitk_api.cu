// splitk_api.cu -- the C ABI of libsplitk (declared in include/splitk.h).
//
// Every entry point validates its arguments completely on the host before any
// CUDA call: the launch contract of the pages "Aligned shared rows for
// pipelined NAX on CUDA" (section "Contract and correctness") and "Wider
// consecutive-weight NAX GEMM" (section "Launch contract and correctness"),
// plus NULL, alignment and aliasing checks on the pointers.  Nothing here
// allocates device memory.

#include <cuda_runtime.h>

#include <algorithm>
#include <vector>
#include <cstdio>

#include "splitk.h"
#include "splitk_internal.h"

namespace splitk {

namespace {
thread_local char g_last_error[256] = "no error";
}

cudaError_t note_error(cudaError_t e, const char *what)
{
    if (e != cudaSuccess)
        std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", what, cudaGetErrorName(e),
                      cudaGetErrorString(e));
    return e;
}

void note_message(const char *what, int code)
{
    std::snprintf(g_last_error, sizeof g_last_error, "%s (code %d)", what, code);
}

const char *last_error_message() { return g_last_error; }

}  // namespace splitk

namespace {

using splitk::GemmProblem;
using splitk::TilePlan;

int geometry_status(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps)
{
    // shape rule: M, K, kps positive multiples of 32; N a positive multiple of 64
    if (M <= 0 || M % 32 || K <= 0 || K % 32 || kps <= 0 || kps % 32 || N <= 0 || N % 64)
        return SPLITK_ERR_SHAPE;
    if (M > SPLITK_MAX_DIM || N > SPLITK_MAX_DIM || K > SPLITK_MAX_DIM) return SPLITK_ERR_SHAPE;
    // split rule: every split starts below K, and together they cover K
    if (S <= 0 || (S - 1) * kps >= K || S * kps < K) return SPLITK_ERR_SPLIT;
    if (S > SPLITK_MAX_SPLITS) return SPLITK_ERR_SPLIT;
    return SPLITK_OK;
}

int elem_bytes(int dtype)
{
    switch (dtype) {
    case SPLITK_F32: return 4;
    case SPLITK_F16: return 2;
    case SPLITK_BF16: return 2;
    default: return 0;
    }
}

struct Range {
    uintptr_t lo, hi;   // [lo, hi)
};

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void *p, uint64_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPLITK_OK : SPLITK_ERR_CUDA; }

// Checks shared by gemm_splitk_bt and gemm_bt.
int validate_gemm(const void *A, const void *B, int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps,
                  int dtype)
{
    int st = geometry_status(M, N, K, S, kps);
    if (st != SPLITK_OK) return st;
    if (elem_bytes(dtype) == 0) return SPLITK_ERR_DTYPE;
    if (!A || !B) return SPLITK_ERR_NULL;
    if (!aligned16(A) || !aligned16(B)) return SPLITK_ERR_ALIGN;
    return SPLITK_OK;
}

// The partial pass into P (and, when `out` is given, the split sum too).
// `prefetch` lets the CTAs that start beside the previous launch prefetch the
// operands into L2.  Only the fused launch uses it: before a partial pass
// there is normally a reduce, which leaves no SM free, and prefetches issued
// once every CTA is running only compete with the loads.  Inside a graph
// capture a launch that may start beside the launch before it, or heads a
// run of launches that may, takes the compact layout (two or three CTAs to
// an SM; the same tiles and sums).  For the partial pass of the two-kernel
// call that took the headline's two-kernel operation from 6.15 to 4.82 us
// per operation on GB300 (graphs of eight; M96 N512 K2048 S4 4.42 -> 3.70).
int run_partial_pass(const void *A, const void *B, float *P, float *out, int64_t M, int64_t N,
                     int64_t K, int64_t S, int64_t kps, int dtype, bool fused, bool prefetch, bool b_kn,
                     cudaStream_t stream)
{
    if (dtype == SPLITK_F32 && b_kn) {   // exact FMA on the CUDA cores
        return cuda_status(splitk::launch_simt_f32(static_cast<const float *>(A), static_cast<const float *>(B), P,
                                                   M, N, K, S, kps, b_kn, stream));
    }
    GemmProblem pr{A, B, P, out, M, N, K, S, kps, dtype == SPLITK_BF16};
    pr.b_kn = b_kn;
    pr.f32 = dtype == SPLITK_F32;   // 3xTF32 on the tensor cores
    const int e = elem_bytes(dtype);
    const splitk::Span reads[2] = {splitk::span_of(A, static_cast<uint64_t>(M * K) * e),
                                   splitk::span_of(B, static_cast<uint64_t>(N * K) * e)};
    splitk::Span writes[2];
    int nw = 0;
    if (P) writes[nw++] = splitk::span_of(P, static_cast<uint64_t>(S * M * N) * 4);
    if (out) writes[nw++] = splitk::span_of(out, static_cast<uint64_t>(M * N) * 4);
    splitk::ChainGuard chain(stream, reads, 2, writes, nw);
    // Inside a capture the launches of a run take the compact layout (two or
    // three CTAs to an SM).  With grouping, a fused run's first launch takes
    // the usual plan instead where the grouped kernels can run it: alone in a
    // graph that is faster, and the next call converts it to the compact plan
    // when it joins (one call per graph on GB300: BF16 M256 N1024 K2048 S2
    // 14.3 -> 10.4 us, M96 N512 K2048 S4 10.5 -> 9.6; graphs of eight and
    // forty unchanged).  A partial pass of the two-kernel call keeps the
    // compact layout: a reduce follows it, so nothing joins it, and the next
    // partial passes share the SMs with it (graphs of eight such calls: 4.89
    // against 5.11 us per call).
    const bool compact = chain.capturing() && (chain.overlap() || chain.fresh());
    TilePlan plan;
    if (compact && !chain.overlap() && fused && splitk::grouping_enabled()) {
        plan = splitk::plan_tc(M, N, K, S, kps, fused, pr.f32, false);
        if (!splitk::head_groupable(pr, plan)) plan = splitk::plan_tc(M, N, K, S, kps, fused, pr.f32, true);
    } else {
        plan = splitk::plan_tc(M, N, K, S, kps, fused, pr.f32, compact, compact && chain.overlap());
    }
    if (!prefetch) plan.prefetchers = 0;
    pr.overlap = chain.overlap();
    pr.store_early = chain.store_early();
    // a call that touches nothing in flight, with the same shape and plan as
    // the launch before it, joins that launch (no node added); the first such
    // call after a run's first launch may convert that launch to its own plan
    int group = 1, mode = pr.overlap ? (pr.store_early ? 2 : 1) : 0;
    bool broken = false;
    if (pr.store_early && splitk::grouping_enabled() &&
        splitk::join_group(pr, plan, chain.capture_id(), chain.dep_node(), &group, &mode, &broken)) {
        chain.commit_joined();
        splitk::note_launch({mode, plan.compact, 1, plan.bn, plan.chunks, plan.stages, plan.kbs,
                             static_cast<int>(plan.smem_bytes), plan.cpc, plan.cluster, group});
        return SPLITK_OK;
    }
    if (broken) {   // the captured graph holds an inconsistent node (last error says which)
        chain.commit(false, false);
        return SPLITK_ERR_CUDA;
    }
    const cudaError_t err = chain.capturing() && splitk::grouping_enabled()
                                ? splitk::launch_tc_grouped(pr, plan, stream, chain.capture_id())
                                : splitk::launch_tc(pr, plan, stream);
    chain.commit(err == cudaSuccess, !pr.overlap);
    splitk::note_launch({mode, plan.compact, chain.capturing() ? 1 : 0, plan.bn, plan.chunks, plan.stages, plan.kbs,
                         static_cast<int>(plan.smem_bytes), plan.cpc, plan.cluster, 1});
    return cuda_status(err);
}

}  // namespace

namespace splitk {

bool batch_possible(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps)
{
    const TilePlan plan = plan_tc(M, N, K, S, kps, true, false, true);
    return plan.compact && plan.split_sum == 2 && !plan.x3 && plan.tile_m == kTileM && plan.bn <= 128 &&
           !plan.rows_first;
}

int run_fused_batch(const void *const *A, const void *const *B, float *const *out, int n, int64_t M, int64_t N,
                    int64_t K, int64_t S, int64_t kps, int dtype, cudaStream_t stream)
{
    if (n < 1 || n > kMaxGroup || dtype == SPLITK_F32 || !fused_in_kernel(M, N, K, S, kps, dtype, false))
        return SPLITK_ERR_CONFIG;
    if (!batch_possible(M, N, K, S, kps)) return SPLITK_ERR_CONFIG;
    const TilePlan plan = plan_tc(M, N, K, S, kps, true, false, true);
    GemmProblem prs[kMaxGroup];
    for (int i = 0; i < n; ++i) prs[i] = GemmProblem{A[i], B[i], nullptr, out[i], M, N, K, S, kps, dtype == SPLITK_BF16};
    const cudaError_t err = launch_tc_batch(prs, n, plan, stream);
    note_launch({0, plan.compact, 0, plan.bn, plan.chunks, plan.stages, plan.kbs, static_cast<int>(plan.smem_bytes),
                 plan.cpc, plan.cluster, n});
    return err == cudaSuccess ? SPLITK_OK : (note_error(err, "batched launch"), SPLITK_ERR_CUDA);
}

}  // namespace splitk

namespace {

// The accumulation pass.  After the partial pass it reads what that pass
// wrote, so it waits for it; a reduce whose partials no running launch
// writes (inside a capture) loads them at once.  It lets the next launch
// start as soon as its own blocks have started (the next partial pass then
// loads under it), except where no run of this library's launches precedes
// it in a capture: there it releases the next launch after its wait and
// heads a new run.
int run_reduce(const float *P, float *out, int64_t S, int64_t M, int64_t N, cudaStream_t stream)
{
    const splitk::Span reads[1] = {splitk::span_of(P, static_cast<uint64_t>(S * M * N) * 4)};
    const splitk::Span writes[1] = {splitk::span_of(out, static_cast<uint64_t>(M * N) * 4)};
    splitk::ChainGuard chain(stream, reads, 1, writes, 1);
    const bool head = chain.capturing() && chain.fresh();
    const cudaError_t err = splitk::launch_reduce(P, out, S, M * N, chain.overlap(), !head, stream);
    chain.commit(err == cudaSuccess, head);
    return cuda_status(err);
}

// The split sum runs inside the tensor-core launch; F32 with the [K,N] weight
// runs on the CUDA cores and always takes the two-kernel path.
bool fused_possible(int dtype, bool b_kn) { return !(dtype == SPLITK_F32 && b_kn); }

}  // namespace

// Whether gemm_bt(fused != 0) sums the splits inside its launch: where the
// tile plan holds all of a tile's splits in one resident cluster.  (F32
// operands with M <= 32 or 8 splits or more once ran the two kernels there,
// which measured faster before the F32 launches grouped; on GB300 the fused
// call now wins for them as well, eagerly (M32 N512 K2048, 2 to 8 splits:
// 9.5 against 11.0-11.3 us; M96 N512 K512 S8 5.5 against 7.4; M256 N1024
// K2048 S8 14.5 both ways) and in graphs of eight (4.1 against 4.9; 2.1
// against 4.0).)
bool splitk::fused_in_kernel(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, int dtype, bool b_kn)
{
    if (!fused_possible(dtype, b_kn)) return false;
    const bool x3 = dtype == SPLITK_F32;
    const TilePlan f = splitk::plan_tc(M, N, K, S, kps, true, x3);
    return f.split_sum == 2;
}

namespace {

size_t partials_bytes(int64_t M, int64_t N, int64_t S) { return static_cast<size_t>(S * M * N) * 4; }

}  // namespace

namespace splitk {

int check_gemm_bt(const void *A, const void *B, const float *out, const void *workspace, size_t workspace_bytes,
                  int64_t M, int64_t N, int64_t K, int64_t splits, int64_t k_per_split, int dtype, int fused)
{
    int st = validate_gemm(A, B, M, N, K, splits, k_per_split, dtype);
    if (st != SPLITK_OK) return st;
    if (fused != 0 && fused != 1 && fused != 3) return SPLITK_ERR_CONFIG;
    if (!out || !workspace) return SPLITK_ERR_NULL;
    if (!aligned16(out) || !aligned16(workspace)) return SPLITK_ERR_ALIGN;
    const size_t ws_need = gemm_bt_workspace_bytes(M, N, K, splits, k_per_split, fused);
    if (workspace_bytes < ws_need) return SPLITK_ERR_WORKSPACE;
    const int e = elem_bytes(dtype);
    const Range ra = range_of(A, static_cast<uint64_t>(M * K) * e);
    const Range rb = range_of(B, static_cast<uint64_t>(N * K) * e);
    const Range ro = range_of(out, static_cast<uint64_t>(M * N) * 4);
    const Range rw = range_of(workspace, ws_need);
    if (overlap(ro, ra) || overlap(ro, rb) || overlap(rw, ra) || overlap(rw, rb) || overlap(rw, ro))
        return SPLITK_ERR_ALIAS;
    return SPLITK_OK;
}

}  // namespace splitk

extern "C" {

int splitk_check_geometry(int64_t M, int64_t N, int64_t K, int64_t splits, int64_t k_per_split)
{
    return geometry_status(M, N, K, splits, k_per_split);
}

static int gemm_splitk_impl(const void *A, const void *B, float *partials, int64_t M, int64_t N, int64_t K,
                            int64_t splits, int64_t k_per_split, int dtype, bool b_kn, void *stream)
{
    int st = validate_gemm(A, B, M, N, K, splits, k_per_split, dtype);
    if (st != SPLITK_OK) return st;
    if (!partials) return SPLITK_ERR_NULL;
    if (!aligned16(partials)) return SPLITK_ERR_ALIGN;
    const int e = elem_bytes(dtype);
    const Range ra = range_of(A, static_cast<uint64_t>(M * K) * e);
    const Range rb = range_of(B, static_cast<uint64_t>(N * K) * e);
    const Range rp = range_of(partials, static_cast<uint64_t>(splits * M * N) * 4);
    if (overlap(rp, ra) || overlap(rp, rb)) return SPLITK_ERR_ALIAS;
    return run_partial_pass(A, B, partials, nullptr, M, N, K, splits, k_per_split, dtype, false, false, b_kn,
                            static_cast<cudaStream_t>(stream));
}

int gemm_splitk_bt(const void *A, const void *B, float *partials, int64_t M, int64_t N, int64_t K, int64_t splits,
                   int64_t k_per_split, int dtype, void *stream)
{
    return gemm_splitk_impl(A, B, partials, M, N, K, splits, k_per_split, dtype, false, stream);
}

int gemm_splitk_kn(const void *A, const void *W, float *partials, int64_t M, int64_t N, int64_t K, int64_t splits,
                   int64_t k_per_split, int dtype, void *stream)
{
    return gemm_splitk_impl(A, W, partials, M, N, K, splits, k_per_split, dtype, true, stream);
}

int splitk_reduce(const float *partials, float *out, int64_t splits, int64_t M, int64_t N, void *stream)
{
    if (M <= 0 || N <= 0 || M > SPLITK_MAX_DIM || N > SPLITK_MAX_DIM) return SPLITK_ERR_SHAPE;
    if (splits <= 0 || splits > SPLITK_MAX_SPLITS) return SPLITK_ERR_SPLIT;
    if (!partials || !out) return SPLITK_ERR_NULL;
    if (!aligned16(partials) || !aligned16(out)) return SPLITK_ERR_ALIGN;
    const Range rp = range_of(partials, static_cast<uint64_t>(splits * M * N) * 4);
    const Range ro = range_of(out, static_cast<uint64_t>(M * N) * 4);
    if (overlap(rp, ro)) return SPLITK_ERR_ALIAS;
    return run_reduce(partials, out, splits, M, N, static_cast<cudaStream_t>(stream));
}

int splitk_prepare_bt(const void *W, void *B, int64_t K, int64_t N, int dtype, void *stream)
{
    // the B that the GEMM's contract accepts: K a positive multiple of 32, N of 64
    if (K <= 0 || K % 32 || N <= 0 || N % 64 || K > SPLITK_MAX_DIM || N > SPLITK_MAX_DIM) return SPLITK_ERR_SHAPE;
    const int e = elem_bytes(dtype);
    if (e == 0) return SPLITK_ERR_DTYPE;
    if (!W || !B) return SPLITK_ERR_NULL;
    if (!aligned16(W) || !aligned16(B)) return SPLITK_ERR_ALIGN;
    const uint64_t bytes = static_cast<uint64_t>(K * N) * e;
    if (overlap(range_of(W, bytes), range_of(B, bytes))) return SPLITK_ERR_ALIAS;
    return cuda_status(splitk::launch_prepare(W, B, K, N, e, static_cast<cudaStream_t>(stream)));
}

size_t gemm_bt_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t splits, int64_t k_per_split, int fused)
{
    (void)fused;
    if (geometry_status(M, N, K, splits, k_per_split) != SPLITK_OK) return 0;
    return partials_bytes(M, N, splits);
}

int gemm_bt_workspace_init(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace) return SPLITK_ERR_NULL;
    if (!aligned16(workspace)) return SPLITK_ERR_ALIGN;
    return cuda_status(splitk::note_error(
        cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)), "cudaMemsetAsync(workspace)"));
}

static int gemm_impl(const void *A, const void *B, float *out, void *workspace, size_t workspace_bytes, int64_t M,
                     int64_t N, int64_t K, int64_t splits, int64_t k_per_split, int dtype, int fused, bool b_kn,
                     void *stream)
{
    int st = splitk::check_gemm_bt(A, B, out, workspace, workspace_bytes, M, N, K, splits, k_per_split, dtype, fused);
    if (st != SPLITK_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float *P = static_cast<float *>(workspace);
    // The fused launch sums the splits inside its clusters.  Where the plan
    // cannot hold a tile's splits in one resident cluster, the call runs the
    // two kernels: summing through global memory instead (arrival counters,
    // the last split reading the others' partials back from L2) measured
    // slower on GB300 than the separate reduce in every such case (BF16 M256
    // N1024 K2048 with 8 splits: 17.9 against 7.0 us).  The chunks do not
    // depend on `fused`, so the result is the same either way, bit for bit.
    if (fused && splitk::fused_in_kernel(M, N, K, splits, k_per_split, dtype, b_kn)) {
        // fused == 1 keeps no partials
        float *keep = fused == 1 ? nullptr : P;
        return run_partial_pass(A, B, keep, out, M, N, K, splits, k_per_split, dtype, true, true, b_kn, s);
    }
    st = run_partial_pass(A, B, P, nullptr, M, N, K, splits, k_per_split, dtype, false, false, b_kn, s);
    if (st != SPLITK_OK) return st;
    return run_reduce(P, out, splits, M, N, s);
}

int gemm_bt(const void *A, const void *B, float *out, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
            int64_t K, int64_t splits, int64_t k_per_split, int dtype, int fused, void *stream)
{
    return gemm_impl(A, B, out, workspace, workspace_bytes, M, N, K, splits, k_per_split, dtype, fused, false, stream);
}

int gemm_bt_batch(const void *const *A, const void *const *B, float *const *out, int64_t count, void *workspace,
                  size_t workspace_bytes, int64_t M, int64_t N, int64_t K, int64_t splits, int64_t k_per_split,
                  int dtype, int fused, void *stream)
{
    if (count < 1 || count > (int64_t(1) << 16) || (fused != 0 && fused != 1)) return SPLITK_ERR_CONFIG;
    if (!A || !B || !out) return SPLITK_ERR_NULL;
    // every operation as gemm_bt would check it, then the outputs against one
    // another, every input and the workspace (sorted ranges: an output may
    // overlap nothing; inputs may overlap inputs)
    std::vector<std::pair<Range, bool>> ranges;   // (bytes, is an output)
    ranges.reserve(static_cast<size_t>(count) * 3 + 1);
    const int e = elem_bytes(dtype);
    for (int64_t i = 0; i < count; ++i) {
        const int st = splitk::check_gemm_bt(A[i], B[i], out[i], workspace, workspace_bytes, M, N, K, splits,
                                             k_per_split, dtype, fused);
        if (st != SPLITK_OK) return st;
        ranges.push_back({range_of(A[i], static_cast<uint64_t>(M * K) * e), false});
        ranges.push_back({range_of(B[i], static_cast<uint64_t>(N * K) * e), false});
        ranges.push_back({range_of(out[i], static_cast<uint64_t>(M * N) * 4), true});
    }
    ranges.push_back({range_of(workspace, gemm_bt_workspace_bytes(M, N, K, splits, k_per_split, fused)), true});
    std::sort(ranges.begin(), ranges.end(),
              [](const std::pair<Range, bool> &x, const std::pair<Range, bool> &y) { return x.first.lo < y.first.lo; });
    // sweep: the furthest end seen so far, and whether an output reaches it
    uint64_t reach = 0, out_reach = 0;
    for (size_t i = 0; i < ranges.size(); ++i) {
        const Range &r = ranges[i].first;
        if (r.hi <= r.lo) continue;
        if (i > 0 && (r.lo < out_reach || (ranges[i].second && r.lo < reach))) return SPLITK_ERR_ALIAS;
        reach = std::max(reach, r.hi);
        if (ranges[i].second) out_reach = std::max(out_reach, r.hi);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool batch = fused == 1 && dtype != SPLITK_F32 &&
                       splitk::fused_in_kernel(M, N, K, splits, k_per_split, dtype, false) &&
                       splitk::batch_possible(M, N, K, splits, k_per_split);
    for (int64_t i = 0; i < count;) {
        const int64_t n = batch ? std::min<int64_t>(count - i, splitk::kMaxGroup) : 1;
        int st;
        if (n > 1) {
            st = splitk::run_fused_batch(A + i, B + i, out + i, static_cast<int>(n), M, N, K, splits, k_per_split,
                                         dtype, s);
        } else {
            st = gemm_impl(A[i], B[i], out[i], workspace, workspace_bytes, M, N, K, splits, k_per_split, dtype, fused,
                           false, stream);
        }
        if (st != SPLITK_OK) return st;
        i += n;
    }
    return SPLITK_OK;
}

int gemm_kn(const void *A, const void *W, float *out, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
            int64_t K, int64_t splits, int64_t k_per_split, int dtype, int fused, void *stream)
{
    return gemm_impl(A, W, out, workspace, workspace_bytes, M, N, K, splits, k_per_split, dtype, fused, true, stream);
}

const char *splitk_last_error(void) { return splitk::last_error_message(); }

int splitk_get_device_status(void *stream)
{
    unsigned status = 0;
    const cudaError_t e = splitk::read_and_clear_device_status(static_cast<cudaStream_t>(stream), &status);
    if (e != cudaSuccess) {
        splitk::note_error(e, "reading the device status word");
        return SPLITK_ERR_CUDA;
    }
    return status ? SPLITK_ERR_DEVICE_TIMEOUT : SPLITK_OK;
}

const char *splitk_status_string(int status)
{
    switch (status) {
    case SPLITK_OK: return "ok";
    case SPLITK_ERR_NULL: return "a required pointer is NULL";
    case SPLITK_ERR_SHAPE: return "M, K and k_per_split must be positive multiples of 32 and N of 64 (within limits)";
    case SPLITK_ERR_SPLIT: return "splits must equal ceil(K / k_per_split): every split starts below K and they cover K";
    case SPLITK_ERR_ALIAS: return "an output range overlaps an input or another output";
    case SPLITK_ERR_ALIGN: return "pointers must be 16-byte aligned";
    case SPLITK_ERR_DTYPE: return "unknown element type";
    case SPLITK_ERR_WORKSPACE: return "workspace smaller than gemm_bt_workspace_bytes()";
    case SPLITK_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case SPLITK_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case SPLITK_ERR_CONFIG: return "invalid configuration value";
    default: return "unknown status";
    }
}

int splitk_set_tile_override(int bn, int chunks, int kblocks_per_stage)
{
    if (bn != 0 && bn != 64 && bn != 128 && bn != 256) return SPLITK_ERR_CONFIG;
    if (chunks != 0 && chunks != 1 && chunks != 2 && chunks != 4 && chunks != 8)
        return SPLITK_ERR_CONFIG;
    if (kblocks_per_stage != 0 && kblocks_per_stage != 1 && kblocks_per_stage != 2 && kblocks_per_stage != 4)
        return SPLITK_ERR_CONFIG;
    splitk::set_tile_override(bn, chunks, kblocks_per_stage);
    return SPLITK_OK;
}

int splitk_describe_launch(int64_t M, int64_t N, int64_t K, int64_t splits, int64_t k_per_split, int dtype, int fused,
                           int *info)
{
    int st = geometry_status(M, N, K, splits, k_per_split);
    if (st != SPLITK_OK) return st;
    if (elem_bytes(dtype) == 0) return SPLITK_ERR_DTYPE;
    if (!info) return SPLITK_ERR_NULL;
    std::fill(info, info + 26, 0);
    const bool x3 = dtype == SPLITK_F32;
    // gemm_bt runs the two kernels where the fused launch could not sum a
    // tile's splits inside one resident cluster
    const bool in_kernel = fused != 0 && splitk::fused_in_kernel(M, N, K, splits, k_per_split, dtype, false);
    const TilePlan p = splitk::plan_tc(M, N, K, splits, k_per_split, in_kernel, x3);
    info[0] = x3 ? 2 : 0;
    info[1] = p.bn;
    info[2] = p.chunks;
    info[3] = p.chunk_len;
    info[4] = p.stages;
    info[5] = p.cluster;
    info[6] = static_cast<int>(p.grid.x);
    info[7] = static_cast<int>(p.grid.y);
    info[8] = static_cast<int>(p.grid.z);
    info[9] = static_cast<int>(p.smem_bytes);
    info[10] = in_kernel ? 1 : 0;
    info[11] = in_kernel ? 1 : 2;
    info[12] = p.kbs;
    info[13] = p.three_d;
    info[14] = p.split_sum;
    info[15] = in_kernel ? p.prefetchers : 0;   // gemm_bt's two-kernel path does not prefetch
    info[16] = p.rows_first;
    info[17] = p.tile_m;
    // the layout a tensor-core launch of this call takes inside a graph
    // capture when it may start beside the launch before it
    {
        const TilePlan c = splitk::plan_tc(M, N, K, splits, k_per_split, in_kernel, x3, true, true);
        info[18] = c.compact;
        info[19] = c.compact ? c.stages : 0;
        info[20] = c.compact ? c.kbs : 0;
        info[21] = c.compact ? static_cast<int>(c.smem_bytes) : 0;
        info[22] = c.compact ? c.cpc : 0;
        info[23] = c.compact ? c.cluster : 0;
        info[24] = c.compact ? static_cast<int>(c.grid.z) : 0;
        info[25] = c.compact ? c.bn : 0;
    }
    return SPLITK_OK;
}

int splitk_set_overlap(int mode)
{
    if (mode < 0 || mode > 2) return SPLITK_ERR_CONFIG;
    splitk::set_overlap_mode(mode);
    return SPLITK_OK;
}

int splitk_last_launch(int *info)
{
    if (!info) return SPLITK_ERR_NULL;
    const splitk::LaunchRecord r = splitk::last_launch();
    info[0] = r.overlap;
    info[1] = r.compact;
    info[2] = r.capturing;
    info[3] = r.bn;
    info[4] = r.chunks;
    info[5] = r.stages;
    info[6] = r.kbs;
    info[7] = r.smem_bytes;
    info[8] = r.cpc;
    info[9] = r.cluster;
    info[10] = r.group;
    return SPLITK_OK;
}

int splitk_selftest_kernel_timeout(const void *A, const void *B, float *out, int64_t M, int64_t N, int64_t K,
                                   int64_t splits, int64_t k_per_split, int dtype, void *stream)
{
    int st = validate_gemm(A, B, M, N, K, splits, k_per_split, dtype);
    if (st != SPLITK_OK) return st;
    if (!out) return SPLITK_ERR_NULL;
    if (!aligned16(out)) return SPLITK_ERR_ALIGN;
    const int e = elem_bytes(dtype);
    const Range ro = range_of(out, static_cast<uint64_t>(M * N) * 4);
    if (overlap(ro, range_of(A, static_cast<uint64_t>(M * K) * e)) ||
        overlap(ro, range_of(B, static_cast<uint64_t>(N * K) * e)))
        return SPLITK_ERR_ALIAS;
    if (!splitk::fused_in_kernel(M, N, K, splits, k_per_split, dtype, false)) return SPLITK_ERR_CONFIG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmProblem pr{A, B, nullptr, out, M, N, K, splits, k_per_split, dtype == SPLITK_BF16};
    pr.f32 = dtype == SPLITK_F32;
    pr.acc_probe = true;
    TilePlan plan = splitk::plan_tc(M, N, K, splits, k_per_split, true, pr.f32);
    plan.prefetchers = 0;
    if (splitk::launch_tc(pr, plan, s) != cudaSuccess) return SPLITK_ERR_CUDA;
    return splitk_get_device_status(stream);
}

int splitk_selftest_bounded_wait(int64_t limit_ns, void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (splitk::launch_wait_selftest(limit_ns, s) != cudaSuccess) return SPLITK_ERR_CUDA;
    return splitk_get_device_status(stream);
}

}  // extern "C"
