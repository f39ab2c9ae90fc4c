// splitk_tc.cu -- the split-K partial pass on the 5th-generation tensor cores.
//
// Computes partials[s,m,n] = sum over split s of A[m,k]*B[n,k] for 16-bit
// operands (BF16 or F16, native, no staging through another type), the
// contract of the pages "Aligned shared rows for pipelined NAX on CUDA" and
// "Wider consecutive-weight NAX GEMM" (sections "Contract and correctness" /
// "Launch contract and correctness").  Optionally the same launch also sums
// the splits into out[m,n] (the pages' separate accumulation pass, fused).
//
// One CTA (128 threads, 4 warps) owns a 128 x BN output tile of one K-chunk:
//   warp 0 lane 0  TMA producer: 128x64 A box + BNx64 B box per stage, both
//                  128-byte swizzled, into a ring of `stages` buffers;
//   warp 1 lane 0  MMA issuer: 4 x tcgen05.mma (M=128, N=BN, K=16) per stage,
//                  accumulating in tensor memory (BN 32-bit columns);
//   all 4 warps    epilogue: tensor memory -> registers -> shared memory
//                  (swizzled 32x32 float boxes), then the tile's F32 sums are
//                  formed and stored with coalesced 16-byte stores.
// A split's K range is cut into `chunks` CTAs; they form a thread-block
// cluster and add their accumulators through distributed shared memory in
// chunk order 0,1,2,..., so the result does not depend on which CTA finishes
// first.  In fused mode the cluster holds every split of the tile and the
// owner of each 16-byte piece also adds the split sums in split order, which
// is exactly what the separate reduce kernel does with the same partials.
//
// Every mbarrier wait has a time limit; on time-out the kernel records a bit
// in g_device_status, drains its own loads in flight, frees its tensor memory
// and finishes without touching the outputs' validity guarantees.

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "splitk_internal.h"

namespace splitk {

__device__ unsigned g_device_status;

namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s; a launch normally takes microseconds
constexpr int kThreads = 128;
constexpr int kMaxCluster = 16;

struct TcArgs {
    float *P;
    float *out;
    int M, N, K, S, kps;
    int chunks, chunk_len, stages, cluster;
    int fused;
    int bf16;
    uint64_t wait_limit_ns;
};

template <int BN>
struct TcShape {
    static constexpr uint32_t kABytes = kTileM * kBlockK * 2;     // 16 KB
    static constexpr uint32_t kBBytes = BN * kBlockK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTmemCols = BN;                     // power of two >= 32
    static constexpr int kPieces = kTileM * BN / 4;               // 16-byte pieces per tile
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_splitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const TcArgs args)
{
    using Sh = TcShape<BN>;
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 1];
    __shared__ uint32_t tmem_slot;
    __shared__ int issued_s, consumed_s;
    __shared__ unsigned abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stages = args.stages;
    const uint32_t base = (ptx::smem_addr(dsmem) + 1023u) & ~1023u;   // swizzle atoms are 1 KB

    const int n_tile = blockIdx.x, m_tile = blockIdx.y;
    const int s = blockIdx.z / args.chunks;
    const int c = blockIdx.z - s * args.chunks;
    const int ks = s * args.kps;
    const int ke = min(ks + args.kps, args.K);            // the last split clamps to K
    const int k_lo = ks + c * args.chunk_len;
    const int k_hi = min(k_lo + args.chunk_len, ke);
    const int klen = k_hi > k_lo ? k_hi - k_lo : 0;       // a chunk past a short split is empty
    const int nkb = (klen + kBlockK - 1) / kBlockK;

    const uint32_t bar0 = ptx::smem_addr(&bars[0]);
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kMaxStages + i); };
    const uint32_t acc_bar = bar0 + 8u * (2 * kMaxStages);

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            ptx::mbar_init(full_bar(i), 1);
            ptx::mbar_init(empty_bar(i), 1);
        }
        ptx::mbar_init(acc_bar, 1);
        issued_s = 0;
        consumed_s = 0;
        abort_s = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(&tmem_slot), Sh::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        const uint64_t pol_a = ptx::l2_policy_evict_last();    // A is re-read by every N tile
        const uint64_t pol_b = ptx::l2_policy_evict_normal();
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int st = kb % stages;
            const uint32_t ph = (kb / stages) & 1;
            if (!ptx::mbar_wait_bounded(empty_bar(st), ph ^ 1u, args.wait_limit_ns)) {
                atomicOr(&abort_s, 1u);
                break;
            }
            const uint32_t sa = base + st * Sh::kStageBytes;
            const int kx = k_lo + kb * kBlockK;
            ptx::mbar_arrive_expect_tx(full_bar(st), Sh::kStageBytes);
            ptx::tma_load_2d(sa, &tmA, full_bar(st), kx, m_tile * kTileM, pol_a);
            ptx::tma_load_2d(sa + Sh::kABytes, &tmB, full_bar(st), kx, n_tile * BN, pol_b);
        }
        issued_s = kb;
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = ptx::idesc_f16_f32acc(args.bf16 != 0, kTileM, BN);
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int st = kb % stages;
            const uint32_t ph = (kb / stages) & 1;
            if (!ptx::mbar_wait_bounded(full_bar(st), ph, args.wait_limit_ns)) {
                atomicOr(&abort_s, 2u);
                break;
            }
            ptx::tc_fence_after_sync();
            const uint32_t sa = base + st * Sh::kStageBytes;
            const uint64_t ad = ptx::sdesc_kmajor_sw128(sa);
            const uint64_t bd = ptx::sdesc_kmajor_sw128(sa + Sh::kABytes);
            const int ksteps = min(kBlockK, klen - kb * kBlockK) / 16;   // 4, or 2 for a 32-long tail
            for (int j = 0; j < ksteps; ++j)   // +32 bytes along K inside the swizzled row
                ptx::mma_f16(tmem, ad + 2u * j, bd + 2u * j, idesc, (kb | j) != 0 ? 1u : 0u);
            ptx::mma_commit(empty_bar(st));    // frees the stage once these MMAs have read it
        }
        consumed_s = kb;
        ptx::mma_commit(acc_bar);              // the accumulator is final
    }
    __syncthreads();

    bool acc_ok = ptx::mbar_wait_bounded(acc_bar, 0, args.wait_limit_ns);
    if (!acc_ok) atomicOr(&abort_s, 4u);
    __syncthreads();
    const bool aborted = abort_s != 0;
    if (aborted && tid == 0) {
        atomicOr(&g_device_status, abort_s);
        for (int kb = consumed_s; kb < issued_s; ++kb)   // loads still in flight into our smem
            ptx::mbar_wait_bounded(full_bar(kb % stages), (kb / stages) & 1, args.wait_limit_ns);
    }
    ptx::tc_fence_after_sync();

    // ---- epilogue 1: tensor memory -> shared memory (reuses the stage ring).
    // Thread (warp w, lane l) holds tile row 32w+l.  Box b = jb*4 + w holds
    // rows 32w..32w+31, columns 32jb..32jb+31 as 32 rows of 128 bytes; the
    // 16-byte piece q of row r sits at position q ^ (r & 7), so the eight
    // threads of a store phase hit eight different bank groups.
    ptx::fence_proxy_async_smem();
    const uint32_t E = base;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const bool have_acc = nkb > 0 && !aborted;
#pragma unroll 1
    for (int jb = 0; jb < BN / 32; ++jb) {
        uint32_t v[32];
        if (have_acc) {
            ptx::tmem_ld_32x32b_x32(lane_base + jb * 32, v);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        const uint32_t row_addr = E + static_cast<uint32_t>(jb * 4 + warp) * 4096u + lane * 128u;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            ptx::st_shared_v4(row_addr + (static_cast<uint32_t>(q ^ (lane & 7)) << 4), v[4 * q],
                              v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        if (!acc_ok) ptx::mbar_wait_bounded(acc_bar, 0, args.wait_limit_ns);
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, Sh::kTmemCols);
    }

    // ---- epilogue 2: sums over the cluster, then coalesced global stores.
    const int Q = args.cluster;
    if (Q > 1) {
        ptx::cluster_arrive();
        ptx::cluster_wait();
    }
    const uint32_t rank = Q > 1 ? ptx::cluster_ctarank() : 0u;
    const int per = (Sh::kPieces + Q - 1) / Q;   // Q = splits*chunks need not be a power of two
    const int g_end = min(Sh::kPieces, static_cast<int>(rank + 1) * per);
    const int row0 = m_tile * kTileM, col0 = n_tile * BN;
    const int C = args.chunks;
    const size_t MN = static_cast<size_t>(args.M) * args.N;
    for (int g = static_cast<int>(rank) * per + tid; g < g_end; g += kThreads) {
        const int b = g >> 8, i = g & 255, rb = i >> 3, j = i & 7;
        const int jb = b >> 2, w = b & 3;
        const uint32_t off = static_cast<uint32_t>(b) * 4096u + rb * 128u + (static_cast<uint32_t>(j ^ (rb & 7)) << 4);
        const int row = row0 + w * 32 + rb;
        const int col = col0 + jb * 32 + j * 4;
        const bool in_rows = row < args.M;
        float4 v[kMaxCluster];
        if (Q == 1) {
            v[0] = ptx::ld_shared_v4(E + off);
        } else {
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (r < Q) v[r] = ptx::ld_cluster_v4(ptx::mapa(E + off, r));
        }
        const size_t elem = static_cast<size_t>(row) * args.N + col;
        if (!args.fused) {
            float4 acc = v[0];
#pragma unroll
            for (int r = 1; r < kMaxCluster; ++r)
                if (r < Q) {
                    acc.x += v[r].x; acc.y += v[r].y; acc.z += v[r].z; acc.w += v[r].w;
                }
            if (in_rows) *reinterpret_cast<float4 *>(args.P + s * MN + elem) = acc;
        } else {
            // rank r = split * C + chunk: close each split's chunk sum, then
            // add the split sums in split order.
            float4 part = make_float4(0.f, 0.f, 0.f, 0.f), tot = part;
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r) {
                if (r < Q) {
                    const int cc = r % C;
                    if (cc == 0) {
                        part = v[r];
                    } else {
                        part.x += v[r].x; part.y += v[r].y; part.z += v[r].z; part.w += v[r].w;
                    }
                    if (cc == C - 1) {
                        const int sp = r / C;
                        if (args.P != nullptr && in_rows)
                            *reinterpret_cast<float4 *>(args.P + sp * MN + elem) = part;
                        if (sp == 0) {
                            tot = part;
                        } else {
                            tot.x += part.x; tot.y += part.y; tot.z += part.z; tot.w += part.w;
                        }
                    }
                }
            }
            if (in_rows) *reinterpret_cast<float4 *>(args.out + elem) = tot;
        }
    }
    if (Q > 1) {   // no CTA leaves while another may still read its shared memory
        ptx::cluster_arrive();
        ptx::cluster_wait();
    }
}

__global__ void wait_selftest_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(a, 1);   // nothing ever arrives on this barrier
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait_bounded(a, 0, limit_ns)) atomicOr(&g_device_status, 8u);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major [rows, K] 16-bit matrix, box = box_rows x 64 elements, 128-byte swizzle.
bool encode_operand(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows, bool bf16)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int g_override_bn = 0, g_override_chunks = 0;

size_t stage_bytes(int bn) { return static_cast<size_t>(kTileM + bn) * kBlockK * 2; }
size_t epi_bytes(int bn) { return static_cast<size_t>(kTileM) * bn * 4; }
constexpr size_t kSmemLimit = 227 * 1024;

template <int BN>
cudaError_t prepare_kernel_attrs()
{
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(tc_splitk_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemLimit));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_splitk_kernel<BN>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
    return cudaSuccess;
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &args, const TilePlan &plan,
                      cudaStream_t stream)
{
    cudaError_t e = prepare_kernel_attrs<BN>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = plan.grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    unsigned nattr = 0;
    if (plan.cluster > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = 1;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = plan.cluster;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, tc_splitk_kernel<BN>, ta, tb, args);
}

int pow2_floor(int64_t x)
{
    int p = 1;
    while (static_cast<int64_t>(p) * 2 <= x) p *= 2;
    return p;
}

}  // namespace

void set_tile_override(int bn, int chunks)
{
    g_override_bn = bn;
    g_override_chunks = chunks;
}

TilePlan plan_tc(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused)
{
    (void)K;
    TilePlan p = {};
    const int64_t mt = (M + kTileM - 1) / kTileM;
    int bn = (N % 128 == 0) ? 128 : 64;
    if (g_override_bn && N % g_override_bn == 0) bn = g_override_bn;
    // Split each split's K range over `chunks` CTAs until the grid roughly
    // fills the GPU (one CTA per SM), keeping chunks of at least 64 elements.
    // The limit on `chunks` does not depend on `fused`, so the fused and the
    // two-kernel paths add the same chunks in the same order.
    const int64_t base = mt * (N / bn) * S;
    int limit = 8;
    if (S <= kMaxCluster) limit = std::min(limit, pow2_floor(kMaxCluster / S));
    int chunks = 1;
    if (g_override_chunks) {
        chunks = std::min(g_override_chunks, limit);
    } else {
        while (chunks * 2 <= limit && base * chunks * 2 <= 160 && kps / (chunks * 2) >= 64) chunks *= 2;
    }
    (void)fused;
    int64_t chunk_len = (kps + chunks - 1) / chunks;
    chunk_len = (chunk_len + 31) / 32 * 32;
    const int64_t nkb = (chunk_len + kBlockK - 1) / kBlockK;
    int max_stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - 1024) / stage_bytes(bn)));
    int stages = static_cast<int>(std::max<int64_t>(2, std::min<int64_t>(nkb, max_stages)));
    p.bn = bn;
    p.chunks = chunks;
    p.chunk_len = static_cast<int>(chunk_len);
    p.stages = stages;
    p.fused = fused ? 1 : 0;
    p.cluster = fused ? static_cast<int>(S) * chunks : chunks;
    p.grid = dim3(static_cast<unsigned>(N / bn), static_cast<unsigned>(mt), static_cast<unsigned>(S * chunks));
    p.smem_bytes = std::max(stages * stage_bytes(bn), epi_bytes(bn)) + 1024;
    return p;
}

cudaError_t launch_tc(const GemmProblem &pr, const TilePlan &plan, cudaStream_t stream)
{
    if (plan.cluster > kMaxCluster || plan.stages > kMaxStages || plan.smem_bytes > kSmemLimit)
        return cudaErrorInvalidConfiguration;
    CUtensorMap ta, tb;
    if (!encode_operand(&ta, pr.A, pr.M, pr.K, kTileM, pr.bf16) ||
        !encode_operand(&tb, pr.B, pr.N, pr.K, plan.bn, pr.bf16))
        return cudaErrorInvalidValue;
    TcArgs a = {};
    a.P = pr.P;
    a.out = pr.out;
    a.M = static_cast<int>(pr.M);
    a.N = static_cast<int>(pr.N);
    a.K = static_cast<int>(pr.K);
    a.S = static_cast<int>(pr.S);
    a.kps = static_cast<int>(pr.kps);
    a.chunks = plan.chunks;
    a.chunk_len = plan.chunk_len;
    a.stages = plan.stages;
    a.cluster = plan.cluster;
    a.fused = plan.fused;
    a.bf16 = pr.bf16 ? 1 : 0;
    a.wait_limit_ns = kWaitLimitNs;
    switch (plan.bn) {
    case 64: return launch_bn<64>(ta, tb, a, plan, stream);
    case 128: return launch_bn<128>(ta, tb, a, plan, stream);
    case 256: return launch_bn<256>(ta, tb, a, plan, stream);
    default: return cudaErrorInvalidConfiguration;
    }
}

cudaError_t read_and_clear_device_status(cudaStream_t stream, unsigned *status)
{
    unsigned zero = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(status, g_device_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned));
}

cudaError_t launch_wait_selftest(int64_t limit_ns, cudaStream_t stream)
{
    limit_ns = std::max<int64_t>(1000, std::min<int64_t>(limit_ns, 1000000000));
    wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(limit_ns));
    return cudaGetLastError();
}

}  // namespace splitk
