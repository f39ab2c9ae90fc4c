// splitk_internal.h -- host-side interfaces between libsplitk's translation
// units (the C-ABI layer in splitk_api.cu and the kernel files).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace splitk {

// What one tensor-core launch computes.
struct GemmProblem {
    const void *A;      // [M,K] row-major, 16-bit elements
    const void *B;      // [N,K] row-major, 16-bit elements; with b_kn, the weight [K,N] row-major
    float *P;           // [S,M,N] partials, or nullptr when not written
    float *out;         // [M,N] sum over splits, or nullptr (two-kernel path)
    int64_t M, N, K, S, kps;
    bool bf16;          // operand type: BF16 (true) or F16 (false)
    bool b_kn = false;  // B given as the [K,N] weight itself (read MN-major)
    bool f32 = false;   // F32 operands: 3xTF32 products on the tensor cores (bf16 ignored)
    bool overlap = false; // no launch that may still run writes A or B: load before the previous grid ends
    bool store_early = false; // (with overlap) none reads or writes P or out either: store before that too
    bool acc_probe = false; // time-out self-test: the wait for the accumulator gives up at once
};

// How it is tiled.  One CTA computes a 128 x bn tile of one K-chunk of one
// split; the `chunks` CTAs of a split (or, when the splits are summed in the
// cluster, all splits * chunks CTAs of the tile) form a thread-block cluster
// and add their accumulators through distributed shared memory, each rank
// owning `share` 16-byte pieces of the tile.
struct TilePlan {
    int bn;             // tile width: 64, 128 or 256
    int chunks;         // CTAs per split along K
    int chunk_len;      // K elements per chunk (multiple of 32)
    int stages;         // shared-memory pipeline depth
    int kbs;            // 64-wide k-blocks per stage
    int three_d;        // stages loaded as one 3-D box per operand (K, kps, chunk_len multiples of 64)
    int cluster;        // CTAs per cluster along grid z (chunks, or splits * chunks)
    int fused;          // this launch also sums over splits
    int split_sum;      // 0 none, 2 inside the cluster (cluster = splits * chunks)
    int share;          // 16-byte pieces of the tile each cluster rank owns
    uint32_t region0;   // bytes of the stage ring / accumulator staging
    int prefetchers;    // CTAs (the first in dispatch order) that prefetch A and B into L2
    int x3;             // F32 operands as 3xTF32: 32-element k-blocks, stages twice the loaded bytes
    int rows_first;     // grid x walks the row tiles, y the column tiles (else x columns, y rows)
    int tile_m;         // rows of A per CTA: 128, or 256 (two accumulators; BN 256, one CTA per tile)
    int compact;        // the ring cut so that two CTAs fit on an SM (same tiles, chunks and sums)
    int recv_in_ring;   // the peers' shares land inside the stage ring once the MMAs are done
    int cpc;            // chunks per CTA: 1, or (merged compact plans) every chunk of the split
    dim3 grid;
    size_t smem_bytes;  // dynamic shared memory per CTA
};

constexpr int kTileM = 128;   // rows per CTA tile (tcgen05 M)
constexpr int kBlockK = 64;   // K elements per pipeline stage: one 128-byte swizzle row
constexpr int kMaxStages = 8;
constexpr int kMaxKbs = 4;     // k-blocks in one pipeline stage (one TMA box per operand)
constexpr int kMaxChunks = 8;  // portable cluster size
constexpr int kMaxGroup = 8;   // independent calls one launch may compute (graph capture)
constexpr size_t kSmemLimit = 226 * 1024;   // dynamic shared memory of a CTA; leaves room for static shared memory

// Whether a CTA with `smem` bytes of dynamic shared memory may allocate `cols`
// tensor-memory columns: the rule that keeps every mix of these kernels'
// CTAs that fits an SM by shared memory within its 512 columns
// (splitk_plan.cu).
bool tmem_fits(int cols, size_t smem);

// Tile choice for a shape (automatic, or the process-wide override).
// x3: F32 operands as 3xTF32 (else 16-bit operands).
// compact: the layout that lets two or three CTAs share an SM, where that
// plan exists (plan.compact says whether it was taken).
// A fused compact plan may give each CTA two consecutive chunks of its split
// (plan.cpc == 2); with whole_k, for a launch that follows another, every
// chunk of every split (plan.cpc > plan.chunks, no cluster) where the
// compact plan would take more than half the SMs.
TilePlan plan_tc(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused, bool x3 = false,
                 bool compact = false, bool whole_k = false);
// The planner's estimate (microseconds) of one tensor-core launch of that
// plan behind another launch, the in-launch split sum included when fused.
double estimate_tc_us(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused, bool x3 = false);
void set_tile_override(int bn, int chunks, int kbs);

// Kernel launches; each returns the launch's CUDA error.
cudaError_t launch_tc(const GemmProblem &p, const TilePlan &plan, cudaStream_t stream);
// The same, inside the capture `capture` (0: not capturing): a launch that
// later calls may join (join_group), where the plan allows grouping.
cudaError_t launch_tc_grouped(const GemmProblem &p, const TilePlan &plan, cudaStream_t stream,
                              unsigned long long capture);
// Whether a launch with this plan can head a group (the grouped kernels
// have an instance for it).
bool head_groupable(const GemmProblem &p, const TilePlan &plan);
// Adds the call to the grouped launch captured as `dep` (the capture's
// current dependency), if it has the same shape and plan and room; returns
// whether it did (and the launch's problem count in *group_size).
bool join_group(const GemmProblem &p, const TilePlan &plan, unsigned long long capture, cudaGraphNode_t dep,
                int *group_size, int *mode, bool *broken);
// One launch computing n (1..kMaxGroup) independent problems of one shape
// with the plan (compact, groupable), outside a capture: the grouped kernel
// with every problem given at once.
cudaError_t launch_tc_batch(const GemmProblem *p, int n, const TilePlan &plan, cudaStream_t stream);
cudaError_t launch_simt_f32(const float *A, const float *B, float *P, int64_t M, int64_t N, int64_t K,
                            int64_t S, int64_t kps, bool b_kn, cudaStream_t stream);
// overlap: nothing that can still be running writes P (splitk_chain.cu);
// release_first: let the next grid start before waiting for the previous one
cudaError_t launch_reduce(const float *P, float *out, int64_t S, int64_t count, bool overlap, bool release_first,
                          cudaStream_t stream);
cudaError_t launch_prepare(const void *W, void *B, int64_t K, int64_t N, int elem_bytes, cudaStream_t stream);

// A byte range [lo, hi) of device memory that a launch reads or writes.
struct Span {
    uintptr_t lo, hi;
};
inline Span span_of(const void *p, uint64_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Span{lo, lo + static_cast<uintptr_t>(bytes)};
}
constexpr int kMaxSpans = 3;

// Decides, for one launch, whether it may load before the previous grid on
// its stream finishes (splitk_chain.cu), and records what it writes.  While a
// capture is active the guard holds the chain table's lock from the decision
// to commit(), so the two see the same chain.
class ChainGuard {
public:
    ChainGuard(cudaStream_t stream, const Span *reads, int n_reads, const Span *writes, int n_writes);
    ChainGuard(const ChainGuard &) = delete;
    ChainGuard &operator=(const ChainGuard &) = delete;
    bool capturing() const { return capturing_; }
    // no launch that may still be running writes what this one reads
    bool overlap() const { return overlap_; }
    // (with overlap) none reads or writes what this one writes either
    bool store_early() const { return store_early_; }
    // the capture, and the node the launch depends on (its chain's last
    // launch, when overlap() holds)
    unsigned long long capture_id() const { return id_; }
    cudaGraphNode_t dep_node() const { return dep_; }
    // no earlier launch of this library precedes it in the capture (or the
    // window was full): a head that independent launches may follow
    bool fresh() const { return fresh_; }
    // after the launch: record its reads and writes (or forget the chain if
    // it failed); `head`: it waited for the previous grid before letting
    // the next one start, so nothing before it can still be running then
    void commit(bool launched, bool head);
    // instead of commit: the call joined the chain's last launch (no node
    // added); its reads and writes are added to that launch's
    void commit_joined();

private:
    cudaStream_t stream_;
    std::unique_lock<std::mutex> lock_;
    unsigned long long id_ = 0;
    bool capturing_ = false, overlap_ = false, fresh_ = false, store_early_ = false;
    cudaGraphNode_t dep_ = nullptr;
    Span reads_[kMaxSpans], writes_[kMaxSpans];
    int n_reads_ = 0, n_writes_ = 0;
};
// 0: every launch waits; 1: overlap in captures; 2: overlap and grouping
void set_overlap_mode(int mode);
bool overlap_enabled();
bool grouping_enabled();

// What the last tensor-core launch of this host thread did (splitk_last_launch).
struct LaunchRecord {
    int overlap, compact, capturing, bn, chunks, stages, kbs, smem_bytes, cpc, cluster, group;
};
void note_launch(const LaunchRecord &r);
LaunchRecord last_launch();

// Whether gemm_bt(fused != 0) sums the splits inside its tensor-core launch
// (else it runs the partial pass and the reduce); dtype as in splitk.h.
bool fused_in_kernel(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, int dtype, bool b_kn);
// n (1..kMaxGroup) fused calls (fused = 1, [N,K] weights) of one shape in one
// launch, where the shape sums its splits inside the launch and its compact
// plan groups; returns SPLITK_ERR_CONFIG, launching nothing, where it does not.
// Arguments as gemm_bt's, already validated, outputs distinct.
int run_fused_batch(const void *const *A, const void *const *B, float *const *out, int n, int64_t M, int64_t N,
                    int64_t K, int64_t S, int64_t kps, int dtype, cudaStream_t stream);
// Whether the 16-bit fused plan of the shape allows such a launch.
bool batch_possible(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps);

// gemm_bt's argument checks (status as gemm_bt returns it; nothing launched),

int check_gemm_bt(const void *A, const void *B, const float *out, const void *workspace, size_t workspace_bytes,
                  int64_t M, int64_t N, int64_t K, int64_t splits, int64_t k_per_split, int dtype, int fused);

// Last-error record (per host thread): what failed and the CUDA error or
// driver result it returned.  note_error passes `e` through.
cudaError_t note_error(cudaError_t e, const char *what);
void note_message(const char *what, int code);
const char *last_error_message();

// Device status word (set by kernels whose bounded waits ran out).
cudaError_t read_and_clear_device_status(cudaStream_t stream, unsigned *status);
cudaError_t launch_wait_selftest(int64_t limit_ns, cudaStream_t stream);

}  // namespace splitk
