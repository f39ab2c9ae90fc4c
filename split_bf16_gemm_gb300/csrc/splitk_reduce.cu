// splitk_reduce.cu -- the accumulation pass: out[i] = sum over s of P[s][i].
//
// The pages run "an existing elementwise accumulation kernel" after the
// partial pass ("Aligned shared rows for pipelined NAX on CUDA", section
// "Contract and correctness"; "Wider consecutive-weight NAX GEMM", section
// "Performance method").  Here it is a memory-bound streaming kernel: each
// thread owns 16-byte pieces of the output, loads the S partial pieces
// (independent 16-byte loads, all in flight together) and adds them in split
// order s = 0, 1, ..., S-1 in F32, starting from P[0] itself.  The grid is a
// multiple of the SM count with a grid-stride loop.  Launched as a
// programmatic dependent of the partial pass: its blocks start while the
// partial pass finishes and wait (griddepcontrol.wait) for it before reading.
// With `release_first` each block lets the next grid start at once (the
// next partial pass then loads its operands while this one sums, where it
// may: splitk_chain.cu); otherwise only after its wait, which makes it the
// head of a run of launches that may overlap.  With `overlap` (no running
// launch writes P) the blocks load at once and wait for the previous grid
// only before their stores.

#include "ptx.cuh"
#include "splitk_internal.h"

namespace splitk {
namespace {

constexpr int kReduceThreads = 256;
constexpr int kUnroll = 8;

__device__ __forceinline__ float4 ld_stream(const float4 *p)
{
    return __ldcs(p);   // partials are read once
}

__global__ void __launch_bounds__(kReduceThreads)
    reduce_v4_kernel(const float4 *__restrict__ P, float4 *__restrict__ out, int S, int64_t n4, int overlap,
                     int release_first)
{
    if (release_first) ptx::launch_dependents();
    if (!overlap) ptx::grid_dependency_wait();   // the partials may be the previous grid's output
    ptx::launch_dependents();                    // (a second invocation changes nothing)
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kReduceThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kReduceThreads + threadIdx.x; i < n4; i += stride) {
        float4 acc = ld_stream(P + i);
        int s = 1;
        for (; s + kUnroll <= S; s += kUnroll) {
            float4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(P + static_cast<int64_t>(s + u) * n4 + i);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
            }
        }
        for (; s < S; ++s) {
            const float4 v = ld_stream(P + static_cast<int64_t>(s) * n4 + i);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (overlap) ptx::grid_dependency_wait();   // the previous grid may still read `out`
        out[i] = acc;
    }
}

// Any element count: the same sums one float at a time.
__global__ void __launch_bounds__(kReduceThreads)
    reduce_scalar_kernel(const float *__restrict__ P, float *__restrict__ out, int S, int64_t n, int overlap,
                         int release_first)
{
    if (release_first) ptx::launch_dependents();
    if (!overlap) ptx::grid_dependency_wait();
    ptx::launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kReduceThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kReduceThreads + threadIdx.x; i < n; i += stride) {
        float acc = P[i];
        for (int s = 1; s < S; ++s) acc += P[static_cast<int64_t>(s) * n + i];
        if (overlap) ptx::grid_dependency_wait();
        out[i] = acc;
    }
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

}  // namespace

cudaError_t launch_reduce(const float *P, float *out, int64_t S, int64_t count, bool overlap, bool release_first,
                          cudaStream_t stream)
{
    static thread_local int sms = 0;
    if (sms == 0) sms = sm_count();
    const bool vec = (count % 4) == 0;
    const int64_t items = vec ? count / 4 : count;
    const int64_t want = (items + kReduceThreads - 1) / kReduceThreads;
    // whole waves of 8 resident blocks per SM at most; a multiple of the SM count
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    int64_t blocks = want < cap ? want : cap;
    if (blocks > sms) blocks = (blocks + sms - 1) / sms * sms;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kReduceThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (vec)
        e = cudaLaunchKernelEx(&cfg, reduce_v4_kernel, reinterpret_cast<const float4 *>(P),
                               reinterpret_cast<float4 *>(out), static_cast<int>(S), items, overlap ? 1 : 0,
                               release_first ? 1 : 0);
    else
        e = cudaLaunchKernelEx(&cfg, reduce_scalar_kernel, P, out, static_cast<int>(S), items, overlap ? 1 : 0,
                               release_first ? 1 : 0);
    if (e != cudaSuccess) return note_error(e, "reduce kernel launch");
    return note_error(cudaGetLastError(), "reduce kernel launch");
}

}  // namespace splitk
