// splitk_internal.h -- host-side interfaces between libsplitk's translation
// units (the C-ABI layer in splitk_api.cu and the kernel files).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace splitk {

// What one tensor-core launch computes.
struct GemmProblem {
    const void *A;      // [M,K] row-major, 16-bit elements
    const void *B;      // [N,K] row-major, 16-bit elements
    float *P;           // [S,M,N] partials, or nullptr when not written
    float *out;         // [M,N] sum over splits, or nullptr (two-kernel path)
    int64_t M, N, K, S, kps;
    bool bf16;          // operand type: BF16 (true) or F16 (false)
};

// How it is tiled.  One CTA computes a 128 x bn tile of one K-chunk of one
// split; `chunks` CTAs share a split, and a thread-block cluster of `cluster`
// CTAs (chunks, or splits*chunks when the kernel also sums the splits) adds
// their accumulators through distributed shared memory.
struct TilePlan {
    int bn;             // tile width: 64, 128 or 256
    int chunks;         // CTAs per split along K
    int chunk_len;      // K elements per chunk (multiple of 32)
    int stages;         // shared-memory pipeline depth
    int cluster;        // CTAs per cluster along grid z
    int fused;          // the cluster also sums over splits
    dim3 grid;
    size_t smem_bytes;  // dynamic shared memory per CTA
};

constexpr int kTileM = 128;   // rows per CTA tile (tcgen05 M)
constexpr int kBlockK = 64;   // K elements per pipeline stage: one 128-byte swizzle row
constexpr int kMaxStages = 8;

// Tile choice for a shape (automatic, or the process-wide override).
TilePlan plan_tc(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused);
void set_tile_override(int bn, int chunks);

// Kernel launches; each returns the launch's CUDA error.
cudaError_t launch_tc(const GemmProblem &p, const TilePlan &plan, cudaStream_t stream);
cudaError_t launch_simt_f32(const float *A, const float *B, float *P, int64_t M, int64_t N, int64_t K,
                            int64_t S, int64_t kps, cudaStream_t stream);
cudaError_t launch_reduce(const float *P, float *out, int64_t S, int64_t count, cudaStream_t stream);

// Device status word (set by kernels whose bounded waits ran out).
cudaError_t read_and_clear_device_status(cudaStream_t stream, unsigned *status);
cudaError_t launch_wait_selftest(int64_t limit_ns, cudaStream_t stream);

}  // namespace splitk
