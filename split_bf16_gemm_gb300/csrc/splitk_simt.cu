// splitk_simt.cu -- the split-K partial pass in exact F32 on the CUDA cores,
// for F32 operands with the [K,N] weight.
//
// One FMA per product, k ascending within the split, F32 accumulator: the
// exact-F32 reference point for the pages' 1e-4 partial tolerance ("Aligned
// shared rows for pipelined NAX on CUDA", section "Contract and
// correctness").  F32 with the prepared [N,K] weight runs on the tensor cores
// as 3xTF32 instead.
//
// Tiling: a 256-thread block owns a 64x64 tile of one split; each thread a
// 4x4 sub-tile.  A and B are staged through shared memory 16 k at a time,
// stored k-major so the inner loop reads broadcast-free rows.  B is either the
// prepared [N,K] weight or the [K,N] weight itself; both fill the same
// shared-memory tile, so the products and their order are the same.

#include "splitk_internal.h"

namespace splitk {
namespace {

constexpr int kT = 64;     // tile rows and columns
constexpr int kKs = 16;    // k per stage
constexpr int kSimtThreads = 256;

// KN: B is the weight W[K,N] itself (element (n,k) at k*N + n), else B[N,K].
template <bool KN>
__global__ void __launch_bounds__(kSimtThreads)
    simt_f32_kernel(const float *__restrict__ A, const float *__restrict__ B, float *__restrict__ P, int M, int N,
                    int K, int kps)
{
    __shared__ float As[kKs][kT + 4];
    __shared__ float Bs[kKs][kT + 4];
    const int s = blockIdx.z;
    const int ks = s * kps;
    const int ke = min(ks + kps, K);   // the last split clamps to K
    const int m0 = blockIdx.y * kT, n0 = blockIdx.x * kT;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = ks; k0 < ke; k0 += kKs) {
        for (int idx = threadIdx.x; idx < kT * kKs; idx += kSimtThreads) {
            const int r = idx / kKs, kk = idx % kKs, k = k0 + kk;
            const int m = m0 + r;
            As[kk][r] = (m < M && k < ke) ? A[static_cast<size_t>(m) * K + k] : 0.f;
            if (!KN) {
                const int n = n0 + r;
                Bs[kk][r] = (n < N && k < ke) ? B[static_cast<size_t>(n) * K + k] : 0.f;
            } else {   // consecutive threads read consecutive n of one W row
                const int kb = idx / kT, c = idx % kT, kw = k0 + kb;
                Bs[kb][c] = (kw < ke) ? B[static_cast<size_t>(kw) * N + n0 + c] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kKs; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *Ps = P + static_cast<size_t>(s) * M * N;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m < M)
            *reinterpret_cast<float4 *>(Ps + static_cast<size_t>(m) * N + n0 + tx * 4) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
}

}  // namespace

cudaError_t launch_simt_f32(const float *A, const float *B, float *P, int64_t M, int64_t N, int64_t K, int64_t S,
                            int64_t kps, bool b_kn, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(N / kT), static_cast<unsigned>((M + kT - 1) / kT), static_cast<unsigned>(S));
    if (b_kn)
        simt_f32_kernel<true><<<grid, kSimtThreads, 0, stream>>>(A, B, P, static_cast<int>(M), static_cast<int>(N),
                                                                static_cast<int>(K), static_cast<int>(kps));
    else
        simt_f32_kernel<false><<<grid, kSimtThreads, 0, stream>>>(A, B, P, static_cast<int>(M), static_cast<int>(N),
                                                                 static_cast<int>(K), static_cast<int>(kps));
    return note_error(cudaGetLastError(), "F32 FMA kernel launch");
}

}  // namespace splitk
