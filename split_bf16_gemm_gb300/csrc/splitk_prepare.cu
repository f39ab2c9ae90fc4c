// splitk_prepare.cu -- weight preparation: B[n,k] = W[k,n].
//
// The pages keep both weight layouts resident and prepare the transposed one
// once, outside timing ("Wider consecutive-weight NAX GEMM", section
// "Performance method": both layouts uploaded once, conversion outside
// timing).  This is that one-shot step on the GPU: a row-major W[K,N] becomes
// the row-major B[N,K] the split-K kernels read.
//
// A memory-bound tiled transpose.  A 256-thread block moves one 64 x 64 tile:
// it reads W's 64 rows with 16-byte loads (coalesced along n), stores them in
// shared memory, and writes B's 64 rows with 16-byte stores (coalesced along
// k).  The element is copied as raw bits, so one kernel serves F16, BF16
// (2 bytes) and F32 (4 bytes).  K is a multiple of 32 and N of 64 (the GEMM
// contract), so only the last k-tile can be half full.

#include "ptx.cuh"
#include "splitk_internal.h"

namespace splitk {
namespace {

constexpr int kTile = 64;
constexpr int kPrepThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kPrepThreads)
    transpose_kernel(const T *__restrict__ W, T *__restrict__ B, int64_t K, int64_t N)
{
    constexpr int kVec = 16 / sizeof(T);                 // elements per 16-byte vector
    constexpr int kVecsPerRow = kTile / kVec;
    // padded by one 32-bit word per row: the column reads spread over the banks
    __shared__ T tile[kTile][kTile + 4 / sizeof(T)];
    ptx::grid_dependency_wait();                         // W may be the previous grid's output
    ptx::launch_dependents();                            // the next launch may start its blocks now
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTile;
    const int64_t k0 = static_cast<int64_t>(blockIdx.y) * kTile;
    // W rows k0..k0+63, columns n0..n0+63  ->  tile[k - k0][n - n0]
    for (int v = threadIdx.x; v < kTile * kVecsPerRow; v += kPrepThreads) {
        const int r = v / kVecsPerRow, c = (v % kVecsPerRow) * kVec;
        if (k0 + r < K) {
            const uint4 x = *reinterpret_cast<const uint4 *>(W + (k0 + r) * N + n0 + c);
            const T *e = reinterpret_cast<const T *>(&x);
#pragma unroll
            for (int i = 0; i < kVec; ++i) tile[r][c + i] = e[i];
        }
    }
    __syncthreads();
    // B rows n0..n0+63, columns k0..k0+63  <-  tile[k - k0][n - n0]
    for (int v = threadIdx.x; v < kTile * kVecsPerRow; v += kPrepThreads) {
        const int r = v / kVecsPerRow, c = (v % kVecsPerRow) * kVec;
        if (k0 + c < K) {                                // K % 32 == 0: whole vectors or none
            uint4 x;
            T *e = reinterpret_cast<T *>(&x);
#pragma unroll
            for (int i = 0; i < kVec; ++i) e[i] = tile[c + i][r];
            *reinterpret_cast<uint4 *>(B + (n0 + r) * K + k0 + c) = x;
        }
    }
}

}  // namespace

cudaError_t launch_prepare(const void *W, void *B, int64_t K, int64_t N, int elem_bytes, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(N / kTile), static_cast<unsigned>((K + kTile - 1) / kTile), 1);
    cfg.blockDim = dim3(kPrepThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (elem_bytes == 2)
        e = cudaLaunchKernelEx(&cfg, transpose_kernel<uint16_t>, static_cast<const uint16_t *>(W),
                               static_cast<uint16_t *>(B), K, N);
    else
        e = cudaLaunchKernelEx(&cfg, transpose_kernel<uint32_t>, static_cast<const uint32_t *>(W),
                               static_cast<uint32_t *>(B), K, N);
    return note_error(e, "weight preparation kernel launch");
}

}  // namespace splitk
