// splitk_tc.cu -- the split-K partial pass on the 5th-generation tensor cores.
//
// Computes partials[s,m,n] = sum over split s of A[m,k]*B[n,k] for 16-bit
// operands (BF16 or F16, native, no staging through another type) and for
// F32 operands as 3xTF32 products (X3), the
// contract of the pages "Aligned shared rows for pipelined NAX on CUDA" and
// "Wider consecutive-weight NAX GEMM" (sections "Contract and correctness" /
// "Launch contract and correctness").  Optionally the same launch also sums
// the splits into out[m,n] (the pages' separate accumulation pass, fused).
//
// One CTA (256 threads, 8 warps) owns a TM x BN output tile of one K-chunk, of
// two consecutive chunks of its split, or (whole-K) of every chunk of every
// split, each chunk in its own accumulator (TM = 128, or 256 as below):
//   thread 0       TMA producer: per stage, kbs 64-wide k-blocks of A (TM
//                  rows) and of B (BN rows), 128-byte swizzled, into a ring
//                  of `stages` buffers; the first stages go out before tensor
//                  memory is allocated;
//   warp 1 lane 0  MMA issuer: tcgen05.mma (M=128, N=BN, K=16; K=8 and three
//                  products per step with X3) from descriptors built once
//                  per stage, accumulating in tensor memory (BN 32-bit
//                  columns per chunk);
//   warps 2-7      before the dependency wait, in the CTAs that start beside
//                  the previous launch: L2 prefetch of this launch's A and B;
//                  with X3, after it: the lo parts of each landed stage;
//   all 8 warps    epilogue: tensor memory -> registers -> shared memory
//                  (swizzled 32x32 float boxes, reusing the stage ring).
// B is either the prepared [N,K] weight (K-major operand) or, with KN, the
// [K,N] weight itself (MN-major operand: boxes of 64 columns by the stage's
// k-rows); both give the same products in the same order.
// 256-row tiles (BN = 256, one CTA per tile, 16-bit operands): each K step is
// two MMAs, rows 0-127 and 128-255 of the stage's A, into two accumulators
// (all 512 tensor-memory columns) with the same B descriptor, and the
// epilogue runs once per 128-row half.  That loads a third fewer bytes per
// product, and launches of many tiles are bound by each SM's TMA intake.
// The grid walks the column tiles first, or the row tiles first where every
// wave would otherwise sweep a B slab too large to stay in L2.
// The CTAs that share a tile (the chunks of a split, or every split and chunk
// of the tile when the launch sums the splits) form one thread-block cluster.
// Each cluster rank owns 1/Q of the tile; each warp pushes the boxes it staged
// to their owners with bulk shared-memory copies (cp.async.bulk into the
// owner's shared memory, counted on the owner's mbarrier), and each owner adds
// the contributions in rank order from its own shared memory -- each split's
// chunks in pairs ((c0 + c1) + (c2 + c3) ...), then the splits in split order,
// the separate reduce kernel's sums -- so the result does not depend on
// arrival order.
//
// Programmatic dependent launch: the kernel waits for the previous grid (whose
// writes it may read) before its first load, and lets the next grid start its
// own set-up once that wait has returned.  With `overlap` the host has
// established that no launch that can still be running writes A or B (the
// chain of launches inside one graph capture, splitk_chain.cu): the loads then
// start at once, the next grid is released at the kernel's start, and the
// wait for the previous grid comes only before the first global store -- or,
// where none of those launches reads or writes this one's outputs either, only
// before one CTA of the grid finishes (the grids still finish in launch
// order).  Consecutive independent operations then run side by side, two or
// three CTAs to an SM in the compact layout (a ring cut to fit, that also
// receives the peers' shares), where a CTA may take two chunks of its split
// or, for large shapes, the whole K range; consecutive calls of one shape may
// also join one launch of the grouped kernel (G problems, found from
// blockIdx.y), whose graph node the host rewrites as calls join it.
//
// Every mbarrier wait has a time limit; on time-out the kernel records a bit
// in g_device_status, drains its own loads in flight, still sends and awaits
// every cluster message (so no peer waits on it), waits for its MMAs, frees
// its tensor memory and finishes; the outputs of that launch are then not
// valid.

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "ptx.cuh"
#include "splitk_internal.h"

namespace splitk {

__device__ unsigned g_device_status;

namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s; a launch normally takes microseconds
constexpr int kThreads = 256;                     // 8 warps: two per tensor-memory lane quarter

// The operands of the problems one launch computes: one, or (G > 1) up to G
// independent problems of the same shape and plan, the group index taken
// from blockIdx.y (blockIdx.y = group * m_tiles + row tile).
template <int G>
struct TcOperands {
    CUtensorMap tm[G][2];       // A and B of each problem
    float *P[G];                // [S,M,N] partials (nullptr: not kept, when the cluster sums the splits)
    float *out[G];              // [M,N], or nullptr when the splits are not summed here
    const uint8_t *A[G], *B[G]; // operands, for the L2 prefetch
};

struct TcArgs {
    int M, N, K, S, kps;
    int group;             // problems in the launch (G > 1 only)
    int m_tiles;           // row tiles of one problem
    int chunks, chunk_len, stages;
    int split_sum;         // 0: none; 2: inside the cluster (cluster = splits x chunks)
    int kbs;               // 64-wide k-blocks per pipeline stage
    int three_d;           // operands loaded as 3-D boxes of kbs k-blocks (else 2-D, kbs == 1)
    int share;             // 16-byte pieces owned by each cluster rank (a multiple of 8)
    uint32_t region0;      // bytes of the stage ring / accumulator staging area
    int bf16;
    uint64_t wait_limit_ns;
    int acc_probe;         // time-out self-test: the wait for the final accumulator gives up at once
    uint64_t a_bytes, b_bytes;
    int prefetchers;       // CTAs, first in dispatch order, that prefetch A and B into L2
    int rows_first;        // blockIdx.x is the row tile and blockIdx.y the column tile
    int overlap;           // 0: wait for the previous grid before the first load; 1: load at once,
                           // wait before the first store; 2: load and store at once, wait
                           // before finishing (no launch in flight reads or writes the outputs)
    int recv_in_ring;      // the peers' shares land in the stage ring, once its MMAs are done
    int cpc;               // chunks per CTA: 1, 2, or (whole-K) every chunk of every split, each in its own accumulator
};

// Part j of `parts` (whole 128-byte lines) of [p, p + bytes) into L2, one
// line per prefetch, spread over threads t = 0..nt-1.  Per-thread prefetches
// keep the TMA unit free for the CTA's own loads.
__device__ __forceinline__ void prefetch_part(const uint8_t *p, uint64_t bytes, int j, int parts, int t, int nt)
{
    const uint64_t part = ((bytes + parts - 1) / parts + 127) & ~uint64_t(127);
    const uint64_t lo = static_cast<uint64_t>(j) * part;
    const uint64_t hi = min(lo + part, bytes);
    for (uint64_t off = lo + static_cast<uint64_t>(t) * 128u; off < hi; off += static_cast<uint64_t>(nt) * 128u)
        ptx::prefetch_l2_line(p + off);
}

// TM: rows of A per CTA.  128 is one MMA's M; 256 (BN = 256 only) is two
// accumulators, rows 0-127 and 128-255, which share every B operand.
template <int BN, int TM = kTileM>
struct TcShape {
    static constexpr uint32_t kABytes = TM * kBlockK * 2;         // one k-block of A: 16 or 32 KB
    static constexpr uint32_t kBBytes = BN * kBlockK * 2;         // one k-block of B
    static constexpr uint32_t kTmemCols = BN * (TM / kTileM);     // power of two >= 32
    static constexpr int kPieces = kTileM * BN / 4;               // 16-byte pieces per 128-row tile
};

// Piece g of the staged tile: 4 consecutive F32 of one row.  Box b = g >> 8
// covers rows 32*(b&3).., columns 32*(b>>2)..; inside it, row rb = (g>>3)&31
// is 128 bytes at (g >> 3) * 128 and holds its 16-byte piece j = g & 7 at
// position j ^ (rb & 7).
struct Piece {
    uint32_t off;   // byte offset in the staging area
    int row, col;   // tile-relative
};

__device__ __forceinline__ Piece piece_at(int g)
{
    const int b = g >> 8, rb = (g >> 3) & 31, j = g & 7;
    Piece p;
    p.off = (static_cast<uint32_t>(g >> 3) << 7) | (static_cast<uint32_t>(j ^ (rb & 7)) << 4);
    p.row = (b & 3) * 32 + rb;
    p.col = (b >> 2) * 32 + j * 4;
    return p;
}

__device__ __forceinline__ void add4(float4 &a, const float4 &b)
{
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// The sum of n (a power of two) consecutive chunk contributions in pairs:
// (v0 + v1) + (v2 + v3), and so on up the tree.  Any aligned run of 2^j
// chunks is a subtree, so a CTA that sums two chunks itself and an owner that
// adds such pair sums give the bits of an owner adding single chunks.
template <int NV>
__device__ __forceinline__ float4 pair_sum(const float4 *v)
{
    if constexpr (NV == 1) {
        return v[0];
    } else {
        float4 a = pair_sum<NV / 2>(v);
        add4(a, pair_sum<NV / 2>(v + NV / 2));
        return a;
    }
}

// The low part of an F32 value for the 3xTF32 products.  The tensor cores
// read an F32 operand as TF32 by dropping its 13 low fraction bits (checked
// on GB300: every output of a one-hot product equals the truncated input), so
// x itself serves as hi = x & ~0x1FFF, and lo = x - hi exactly (at most 13
// significant bits, of which the tensor cores keep the top 11).  Non-finite
// values get lo = 0.
__device__ __forceinline__ uint32_t tf32_lo(uint32_t x)
{
    if ((x & 0x7F800000u) == 0x7F800000u) return 0u;
    return __float_as_uint(__uint_as_float(x) - __uint_as_float(x & 0xFFFFE000u));
}

// The owner's sums when the cluster holds every split of the tile (rank =
// split * CC + chunk): each split's chunks in pairs (pair_sum), then the
// splits in split order -- the additions the reduce kernel makes on the same
// partials, which are also stored with HAS_P.  rbase[r] plus a piece's staging offset
// addresses rank r's contribution to it.  The chunk count and HAS_P are
// template parameters so that the grouping costs no branches: decided at run
// time, the branches of this short sequence (resolved one after another in
// every warp) about doubled the loop's time.  Each thread loads both of its
// pieces (2 x Q float4) before it adds and stores.
template <int Q, int CC, bool HAS_P>
__device__ __forceinline__ void cluster_split_sum(const uint32_t (&rbase)[Q], int g_lo, int g_hi, int rows_here,
                                                  size_t tile0, int N, size_t MN, float *P, float *out)
{
    static_assert(Q % CC == 0, "the cluster holds whole splits");
    auto finish = [&](const Piece &p, const float4 (&v)[Q]) {
        const size_t e = tile0 + static_cast<size_t>(p.row) * N + p.col;
        const bool live = p.row < rows_here;
        float4 tot = v[0];
#pragma unroll
        for (int sp = 0; sp < Q / CC; ++sp) {
            const float4 part = pair_sum<CC>(&v[sp * CC]);
            if (HAS_P && live) *reinterpret_cast<float4 *>(P + sp * MN + e) = part;
            if (sp == 0)
                tot = part;
            else
                add4(tot, part);
        }
        if (live) *reinterpret_cast<float4 *>(out + e) = tot;
    };
    for (int g0 = g_lo; g0 < g_hi; g0 += 2 * kThreads) {
        const int g1 = g0 + kThreads;
        const Piece p0 = piece_at(g0), p1 = piece_at(min(g1, g_hi - 1));
        float4 v0[Q], v1[Q];
#pragma unroll
        for (int r = 0; r < Q; ++r) v0[r] = ptx::ld_shared_v4(rbase[r] + p0.off);
#pragma unroll
        for (int r = 0; r < Q; ++r) v1[r] = ptx::ld_shared_v4(rbase[r] + p1.off);
        finish(p0, v0);
        if (g1 < g_hi) finish(p1, v1);
    }
}

template <int Q, bool HAS_P>
__device__ __forceinline__ void cluster_split_sum_for(int C, const uint32_t (&rbase)[Q], int g_lo, int g_hi,
                                                      int rows_here, size_t tile0, int N, size_t MN, float *P,
                                                      float *out)
{
    // the chunks of a split: a power of two dividing Q (the host checks this
    // before the launch; anything else would leave `out` unwritten, so it
    // is reported in the status word rather than skipped silently)
    if (C == 1) {
        cluster_split_sum<Q, 1, HAS_P>(rbase, g_lo, g_hi, rows_here, tile0, N, MN, P, out);
        return;
    }
    if constexpr (Q % 2 == 0) {
        if (C == 2) {
            cluster_split_sum<Q, 2, HAS_P>(rbase, g_lo, g_hi, rows_here, tile0, N, MN, P, out);
            return;
        }
    }
    if constexpr (Q % 4 == 0) {
        if (C == 4) {
            cluster_split_sum<Q, 4, HAS_P>(rbase, g_lo, g_hi, rows_here, tile0, N, MN, P, out);
            return;
        }
    }
    if constexpr (Q % 8 == 0) {
        if (C == 8) {
            cluster_split_sum<Q, 8, HAS_P>(rbase, g_lo, g_hi, rows_here, tile0, N, MN, P, out);
            return;
        }
    }
    atomicOr(&g_device_status, 64u);
}

// KN: B is the [K,N] weight (MN-major operand).  X3: F32 operands, each
// product formed as three TF32 products (hi*lo + lo*hi + hi*hi).  TM: rows
// of A per CTA; 256 only for 16-bit operands, BN = 256 and one CTA per tile
// that keeps or sums its own partials (no cluster).
// Registers: at most 85 per thread for clusters of up to 4 (three CTAs per
// SM in the compact layout), else 128 (two); no instantiation spills.
template <int BN, int Q, bool KN, bool X3, int TM = kTileM, int G = 1>
__global__ void __launch_bounds__(kThreads, Q <= 4 ? 3 : 2)
    tc_splitk_kernel(const __grid_constant__ TcOperands<G> ops, const TcArgs args)
{
    static_assert(!(KN && X3), "F32 operands with the [K,N] weight run on the CUDA cores");
    static_assert(TM == kTileM || (TM == 2 * kTileM && BN == 256 && Q == 1 && !X3), "256-row tiles");
    constexpr int KB = X3 ? 32 : kBlockK;          // k elements per 128-byte swizzle row
    constexpr int KSTEP = X3 ? 8 : 16;             // k per MMA instruction
    constexpr int kHalves = TM / kTileM;           // accumulators (128-row halves of the tile)
    using Sh = TcShape<BN, TM>;
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t bars[3 * kMaxStages + 2];
    __shared__ uint32_t tmem_slot;
    __shared__ int issued_s, consumed_s;
    __shared__ unsigned abort_s;

    // An overlapping launch lets the next grid start at once: its CTAs then
    // take the slots that free up while this grid runs.  (On GB300 the
    // headline shape went from 3.84 to 3.60 us per operation in graphs of
    // eight against releasing after the set-up.)
    if (args.overlap) ptx::launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stages = args.stages;
    const uint32_t raw = ptx::smem_addr(dsmem);
    const uint32_t base = (raw + 1023u) & ~1023u;   // swizzle atoms are 1 KB
    const uint32_t E = base;                        // accumulator staging, over the ring
    // the peers' shares of this CTA's pieces: after the staging area, inside the
    // ring (free once the MMAs are done), or after the ring
    const uint32_t recv = base + (args.recv_in_ring ? static_cast<uint32_t>(kTileM * BN * 4) : args.region0);

    const int n_tile = args.rows_first ? blockIdx.y : blockIdx.x;
    int m_tile = args.rows_first ? blockIdx.x : blockIdx.y;
    int grp = 0;                                    // the problem (grouped launches walk columns first)
    if constexpr (G > 1) {
        grp = m_tile / args.m_tiles;
        m_tile -= grp * args.m_tiles;
    }
    const CUtensorMap *const tmA = &ops.tm[grp][0];
    const CUtensorMap *const tmB = &ops.tm[grp][1];
    float *const P = ops.P[grp];
    float *const out = ops.out[grp];
    // A CTA covers cpc consecutive (split, chunk) units, each summed in its
    // own accumulator (cpc > 1 only for 128-row plans whose chunks are whole
    // k-blocks of whole stages): one chunk, two chunks or every chunk of a
    // split, or (whole_k) every chunk of every split, where the splits are
    // full and their chunks tile them.  The same products, chunk sums and
    // order as one CTA per chunk: the chunk sums (and with whole_k the split
    // sum) are taken before the exchange.  CC CTAs cover a split.
    const int cpc = args.cpc;
    const int C = args.chunks;
    // (whole_k only in the kernels a whole-K plan launches: 16-bit, 128 x 128
    // tiles, no cluster; the others keep their registers)
    constexpr bool kWholeK = Q == 1 && BN == 128 && !X3 && TM == kTileM;
    const bool whole_k = kWholeK && cpc > C;
    const int CC = whole_k ? 1 : C / cpc;
    const int u0 = static_cast<int>(blockIdx.z) * cpc;
    const int s = u0 / C;                           // its first split
    const int c = u0 - s * C;                       // its first chunk there
    const int rank = static_cast<int>(blockIdx.z) % Q;  // in the 1 x 1 x Q cluster: split*CC + CTA of the split
    const int ks = s * args.kps;
    const int ke = whole_k ? args.K : min(ks + args.kps, args.K);   // the last split clamps to K
    const int k_lo = ks + c * args.chunk_len;
    const int k_hi = min(k_lo + cpc * args.chunk_len, ke);
    const int klen = k_hi > k_lo ? k_hi - k_lo : 0; // a chunk past a short split is empty
    const int nkb = (klen + KB - 1) / KB;
    const int share = args.share;
    const int my_lo = min(Sh::kPieces, rank * share);
    const int my_hi = min(Sh::kPieces, my_lo + share);

    const uint32_t bar0 = ptx::smem_addr(&bars[0]);
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kMaxStages + i); };
    const uint32_t acc_bar = bar0 + 8u * (2 * kMaxStages);
    const uint32_t recv_bar = bar0 + 8u * (2 * kMaxStages + 1);
    auto conv_bar = [&](int i) { return bar0 + 8u * (2 * kMaxStages + 2 + i); };   // X3: stage split

    // Stage i holds k-blocks i*kbs .. i*kbs+kbs-1 of the chunk: kbs slabs of A
    // (128 rows x 128 bytes each) then kbs slabs of B (BN rows x 128 bytes).
    // With X3 the loaded half serves as the hi parts as it is and a second
    // half of the same layout holds the lo parts.
    const int kbs = args.kbs;
    const uint32_t load_bytes = static_cast<uint32_t>(kbs) * (Sh::kABytes + Sh::kBBytes);
    const uint32_t stage_bytes = X3 ? 2u * load_bytes : load_bytes;
    const int nstg = (nkb + kbs - 1) / kbs;
    const int pre = min(stages, nstg);              // stages that need no free slot
    auto issue_stage = [&](int i, int slot) {
        const uint32_t sa = base + slot * stage_bytes;
        const uint32_t bar = full_bar(slot);
        ptx::mbar_arrive_expect_tx(bar, load_bytes);
        if (args.three_d) {                         // one box per operand: kbs k-blocks at once
            const int kb = k_lo / KB + i * kbs;
            ptx::tma_load_3d(sa, tmA, bar, 0, m_tile * TM, kb, ptx::l2_policy_evict_last());
            if constexpr (!KN)
                ptx::tma_load_3d(sa + kbs * Sh::kABytes, tmB, bar, 0, n_tile * BN, kb,
                                 ptx::l2_policy_evict_normal());
        } else {                                    // kbs == 1
            const int kx = k_lo + i * KB;
            ptx::tma_load_2d(sa, tmA, bar, kx, m_tile * TM, ptx::l2_policy_evict_last());
            if constexpr (!KN)
                ptx::tma_load_2d(sa + Sh::kABytes, tmB, bar, kx, n_tile * BN, ptx::l2_policy_evict_normal());
        }
        if constexpr (KN) {
            // the [K,N] weight: BN/64 boxes of 64 columns x kbs*64 k-rows
            // (128-byte rows, N contiguous), one after another
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
                ptx::tma_load_2d(sa + kbs * Sh::kABytes + static_cast<uint32_t>(j * kbs) * 8192u, tmB, bar,
                                 n_tile * BN + j * 64, k_lo + i * kbs * kBlockK, ptx::l2_policy_evict_normal());
        }
    };
    if (tid == 0) {
        // the tensor maps first: the first load waits for their fetch
        ptx::prefetch_tensormap(tmA);
        ptx::prefetch_tensormap(tmB);
        for (int i = 0; i < stages; ++i) {
            ptx::mbar_init(full_bar(i), 1);
            ptx::mbar_init(empty_bar(i), 1);
            if (X3) ptx::mbar_init(conv_bar(i), kThreads / 32 - 2);   // one arrival per converting warp
        }
        ptx::mbar_init(acc_bar, 1);
        ptx::mbar_init(recv_bar, 1);
        issued_s = 0;
        consumed_s = 0;
        abort_s = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
        const uint32_t incoming = static_cast<uint32_t>((Q - 1) * (my_hi - my_lo)) * 16u;
        if (incoming)
            ptx::mbar_arrive_expect_tx(recv_bar, incoming);
        else
            ptx::mbar_arrive(recv_bar);
        if (!args.overlap) {
            ptx::grid_dependency_wait();   // A and B may be the previous grid's output
            // the previous grid has finished: the next one may start (this
            // thread's release counts for the CTA; the others' below are no-ops)
            ptx::launch_dependents();
        }
        for (int i = 0; i < pre; ++i) issue_stage(i, i);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(&tmem_slot), Sh::kTmemCols * static_cast<uint32_t>(cpc));
        ptx::tmem_relinquish();
    }
    if (warp >= 2) {
        // CTAs that start while the previous grid still runs (the first ones
        // dispatched, on the SMs it leaves free) bring this launch's operands
        // into L2 for everyone.  L2 is the point of coherence, so a line
        // fetched before the previous grid writes it is updated, never stale.
        const int disp = (blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * (blockIdx.z / Q))) * Q +
                         static_cast<int>(blockIdx.z % Q);
        if (disp < args.prefetchers) {
            prefetch_part(ops.A[grp], args.a_bytes, disp, args.prefetchers, tid - 64, kThreads - 64);
            prefetch_part(ops.B[grp], args.b_bytes, disp, args.prefetchers, tid - 64, kThreads - 64);
        }
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    // the barrier inits were published by thread 0's fence.mbarrier_init; the
    // arrival itself needs no release semantics.  With the receive slots in
    // the ring, this CTA arrives only once its MMAs have read the ring.
    if (Q > 1 && !args.recv_in_ring) ptx::cluster_arrive_relaxed();
    // Without overlap the next grid is released after the wait (an
    // overlapping launch released it at its start; a second release is a
    // no-op).  (Written as one conditional wait and an unconditional
    // release: the same choice as two branches measured 0.1-0.4 us slower
    // per launch on GB300, in both modes.)
    if (!args.overlap) ptx::grid_dependency_wait();
    ptx::launch_dependents();
    const uint32_t tmem = tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: the stages that had to wait for a free slot.
        // Slot and phase advance by counting (no division per stage: the
        // loops below are on the path from a landing to the next load).
        int i = pre;
        int st = pre == stages ? 0 : pre;
        uint32_t ph = pre == stages ? 1u : 0u;
        for (; i < nstg; ++i) {
            if (!ptx::mbar_wait_bounded(empty_bar(st), ph ^ 1u, args.wait_limit_ns)) {
                atomicOr(&abort_s, 1u);
                break;
            }
            issue_stage(i, st);
            if (++st == stages) {
                st = 0;
                ph ^= 1u;
            }
        }
        issued_s = i;
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer.  A single thread issues every MMA, and no other
        // warp hides its scalar latency, so each tcgen05.mma must cost as few
        // dependent instructions as possible: the stage's descriptors are
        // built once, and each operand slice is reached by adding a constant
        // to the descriptor's low word.  Its start-address field (bits 0-13,
        // bytes >> 4) is the low end of that word and every shared-memory
        // address is below 256 KB, so the addition never carries out of the
        // field.  The k-blocks of a stage (at most kMaxKbs) and the K steps
        // of a k-block are unrolled.  (A rolled loop with the descriptors
        // rebuilt per MMA issued the 32 MMAs of a 128 x 64 x 512 chunk in
        // about 3,600 cycles, against about 2,100 for the tensor core to run
        // them.)
        const uint32_t idesc = X3 ? ptx::idesc_tf32_f32acc(kTileM, BN)
                                  : ptx::idesc_f16_f32acc(args.bf16 != 0, kTileM, BN, KN);
        const uint32_t b_lbo = static_cast<uint32_t>(kbs) * 8192u;   // [K,N]: next 64 columns
        const uint32_t lo_half = load_bytes >> 4;                     // X3: the lo parts, in descriptor units
        const bool short_tail = (klen % KB) != 0;   // a 2-D 16-bit chunk may end in a 32-long k-block
        const int kpc = args.chunk_len / KB;        // k-blocks per chunk (a multiple of kbs when cpc > 1)
        // one K step of k-block slice (a, b) (low descriptor words)
        auto issue = [&](uint32_t d, uint32_t a, uint32_t b, uint32_t ahi, uint32_t bhi, int k, uint32_t accumulate) {
            if constexpr (X3) {
                // the small products first, then hi*hi; +32 bytes (8 F32) along K per step
                ptx::mma_tf32(d, ptx::desc64(a + 2u * k, ahi), ptx::desc64(b + lo_half + 2u * k, bhi), idesc,
                              accumulate);
                ptx::mma_tf32(d, ptx::desc64(a + lo_half + 2u * k, ahi), ptx::desc64(b + 2u * k, bhi), idesc, 1u);
                ptx::mma_tf32(d, ptx::desc64(a + 2u * k, ahi), ptx::desc64(b + 2u * k, bhi), idesc, 1u);
            } else {
                // A: +32 bytes along K inside its swizzled rows.  B: the same,
                // or for the [K,N] weight 16 k-rows of 128 bytes further (2 KB)
                const uint32_t bk = b + (KN ? 128u : 2u) * k;
                ptx::mma_f16(d, ptx::desc64(a + 2u * k, ahi), ptx::desc64(bk, bhi), idesc, accumulate);
                if constexpr (TM == 2 * kTileM)   // rows 128-255: 16 KB further, the second accumulator
                    ptx::mma_f16(d + BN, ptx::desc64(a + 1024u + 2u * k, ahi), ptx::desc64(bk, bhi), idesc,
                                 accumulate);
            }
        };
        int i = 0, st = 0;
        uint32_t ph = 0;
        int jc = 0, kb_in = 0;   // cpc > 1: the chunk (accumulator) of the stage, its first k-block in it
        for (; i < nstg; ++i) {
            if (!ptx::mbar_wait_bounded(X3 ? conv_bar(st) : full_bar(st), ph, args.wait_limit_ns)) {
                atomicOr(&abort_s, 2u);
                break;
            }
            ptx::tc_fence_after_sync();
            const uint32_t sa = base + st * stage_bytes;
            const uint32_t sb = sa + kbs * Sh::kABytes;
            const uint64_t a0 = ptx::sdesc_kmajor_sw128(sa);
            const uint64_t b0 = KN ? ptx::sdesc_mnmajor_sw128(sb, b_lbo) : ptx::sdesc_kmajor_sw128(sb);
            const uint32_t alo = static_cast<uint32_t>(a0), ahi = static_cast<uint32_t>(a0 >> 32);
            const uint32_t blo = static_cast<uint32_t>(b0), bhi = static_cast<uint32_t>(b0 >> 32);
            const int kb0 = i * kbs;
            const int nk = min(kbs, nkb - kb0);
            // the chunk's first MMA starts its accumulator
            const uint32_t d = tmem + static_cast<uint32_t>(jc * BN);
            uint32_t accumulate = (cpc > 1 ? kb_in : i) > 0 ? 1u : 0u;
            if (cpc > 1 && (kb_in += kbs) == kpc) {
                kb_in = 0;
                ++jc;
            }
#pragma unroll
            for (int j = 0; j < kMaxKbs; ++j) {
                if (j >= nk) break;
                const uint32_t a = alo + static_cast<uint32_t>(j) * (Sh::kABytes >> 4);
                const uint32_t b = blo + static_cast<uint32_t>(j) * ((KN ? 8192u : Sh::kBBytes) >> 4);
                if (short_tail && kb0 + j == nkb - 1) {
                    // the 32-long tail: exactly two K steps (chunk lengths
                    // are multiples of 32, so only a 16-bit 2-D chunk has
                    // one).  The count is a constant on purpose: the same
                    // two MMAs in a loop bounded by (klen % KB) / KSTEP
                    // contributed only the first K step on GB300.
#pragma unroll
                    for (int k = 0; k < KB / KSTEP / 2; ++k) {
                        issue(d, a, b, ahi, bhi, k, accumulate);
                        accumulate = 1u;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < KB / KSTEP; ++k) {
                        issue(d, a, b, ahi, bhi, k, accumulate);
                        accumulate = 1u;
                    }
                }
            }
            ptx::mma_commit(empty_bar(st));    // frees the slot once these MMAs have read it
            if (++st == stages) {
                st = 0;
                ph ^= 1u;
            }
        }
        consumed_s = i;
        ptx::mma_commit(acc_bar);              // the accumulator is final
    } else if (X3 && warp >= 2) {
        // ---- converters (warps 2-7): the lo parts of each landed stage go to
        // the second half, then the stage is handed to the MMA issuer
        const int t = tid - 64;
        int st = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nstg; ++i) {
            if (!ptx::mbar_wait_bounded(full_bar(st), ph, args.wait_limit_ns)) {
                atomicOr(&abort_s, 8u);
                break;
            }
            const uint32_t sa = base + st * stage_bytes;
            // four 16-byte pieces per thread at a time: their loads are issued
            // before any of their stores (the shared-memory accesses are
            // ordered asm, so one piece at a time would wait out each load)
            constexpr uint32_t kStep = (kThreads - 64) * 16u;
            constexpr int kBatch = 4;
            auto convert_store = [&](uint32_t off, const float4 &v) {
                ptx::st_shared_v4(sa + load_bytes + off, tf32_lo(__float_as_uint(v.x)), tf32_lo(__float_as_uint(v.y)),
                                  tf32_lo(__float_as_uint(v.z)), tf32_lo(__float_as_uint(v.w)));
            };
            uint32_t off = static_cast<uint32_t>(t) * 16u;
            for (; off + (kBatch - 1) * kStep < load_bytes; off += kBatch * kStep) {
                float4 v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) v[u] = ptx::ld_shared_v4(sa + off + u * kStep);
#pragma unroll
                for (int u = 0; u < kBatch; ++u) convert_store(off + u * kStep, v[u]);
            }
            for (; off < load_bytes; off += kStep) convert_store(off, ptx::ld_shared_v4(sa + off));
            ptx::fence_proxy_async_smem();     // the tensor cores read what these threads wrote
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(conv_bar(st));
            if (++st == stages) {
                st = 0;
                ph ^= 1u;
            }
        }
    }
    // time-out self-test: the warps that wait for the accumulator and take no
    // part in the main loop (2-7) test it once, before the MMA issuer has
    // finished, and give up as a wait that ran out would
    if (args.acc_probe && warp >= 2 && !ptx::mbar_test_wait(acc_bar, 0)) atomicOr(&abort_s, 4u);
    __syncthreads();

    const bool acc_ok = ptx::mbar_wait_bounded(acc_bar, 0, args.wait_limit_ns);
    if (!acc_ok) atomicOr(&abort_s, 4u);
    __syncthreads();
    const bool aborted = abort_s != 0;
    if (aborted && tid == 0) {
        atomicOr(&g_device_status, abort_s);
        const int issued = max(issued_s, pre);
        for (int i = consumed_s; i < issued; ++i)      // loads still in flight into our smem
            ptx::mbar_wait_bounded(full_bar(i % stages), (i / stages) & 1, args.wait_limit_ns);
    }
    ptx::tc_fence_after_sync();
    // the ring is free (every stage landed and was read by the MMAs, or was
    // drained above): the peers may push into the receive slots inside it
    if (Q > 1 && args.recv_in_ring) ptx::cluster_arrive_relaxed();

    // ---- epilogue 1: tensor memory -> staging.  Warp w reads lane quarter
    // q = w % 4 (tile rows 32q..32q+31, one per thread) and column half w / 4;
    // the eight threads of a store phase hit eight bank groups.
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool have_acc = nkb > 0 && !aborted;
    // With two accumulators (TM = 256) the staging, the stores and the sums
    // below run once per 128-row half, the second after the first's stores
    // have read the staging.
#pragma unroll 1
    for (int h = 0; h < kHalves; ++h) {
        if (h > 0) __syncthreads();
#pragma unroll 1
        for (int jb = half * (BN / 64); jb < (half + 1) * (BN / 64); ++jb) {
            const uint32_t row_addr = E + static_cast<uint32_t>(jb * 4 + quarter) * 4096u + lane * 128u;
            if (cpc == 1) {
                uint32_t v[32];
                if (have_acc) {
                    ptx::tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(h * BN + jb * 32), v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    ptx::st_shared_v4(row_addr + (static_cast<uint32_t>(q ^ (lane & 7)) << 4), v[4 * q],
                                      v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
                if (!whole_k) {
                    // the chunk sum of a pair (cpc is 2 here): chunk 0 + chunk 1,
                    // a chunk past the split's end adding +0 -- the pair sum
                    // the owner adds when each chunk has its own CTA.  16
                    // columns at a time.
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[16];
                        const uint32_t col = static_cast<uint32_t>(jb * 32 + hh * 16);
                        if (have_acc) {
                            ptx::tmem_ld_32x32b_x16(lane_base + col, v);
#pragma unroll 1
                            for (int j = 1; j < cpc; ++j) {
                                uint32_t w[16];
                                if (k_lo + j * args.chunk_len < k_hi) {
                                    ptx::tmem_ld_32x32b_x16(lane_base + static_cast<uint32_t>(j * BN) + col, w);
                                } else {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) w[i] = 0u;
                                }
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(w[i]));
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = 0u;
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ptx::st_shared_v4(row_addr + (static_cast<uint32_t>((hh * 4 + q) ^ (lane & 7)) << 4),
                                              v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    }
                } else {
                    // whole_k: each split's chunk sum as above (stored as the
                    // split's partials where they are kept), then the splits
                    // in split order, the owner's sums.
                    const int sps = cpc / C;                  // splits the CTA covers
                    const int cps = C;                        // their chunks
                    const int prow = quarter * 32 + lane;     // this thread's tile row
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[16];
                        const uint32_t col = static_cast<uint32_t>(jb * 32 + hh * 16);
#pragma unroll 1
                        for (int sp = 0; sp < sps; ++sp) {
                            uint32_t w[16];
#pragma unroll 1
                            for (int j = 0; j < cps; ++j) {
                                const int a = sp * cps + j;
                                uint32_t x[16];
                                if (have_acc && k_lo + a * args.chunk_len < k_hi) {
                                    ptx::tmem_ld_32x32b_x16(lane_base + static_cast<uint32_t>(a * BN) + col, x);
                                } else {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) x[i] = 0u;
                                }
                                if (j == 0) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) w[i] = x[i];
                                } else {
#pragma unroll
                                    for (int i = 0; i < 16; ++i)
                                        w[i] = __float_as_uint(__uint_as_float(w[i]) + __uint_as_float(x[i]));
                                }
                            }
                            if (P != nullptr && prow < args.M - m_tile * TM) {
                                float *dst = P + static_cast<size_t>(s + sp) * args.M * args.N +
                                             static_cast<size_t>(m_tile * TM + prow) * args.N + n_tile * BN + col;
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    *reinterpret_cast<float4 *>(dst + 4 * q) =
                                        make_float4(__uint_as_float(w[4 * q]), __uint_as_float(w[4 * q + 1]),
                                                    __uint_as_float(w[4 * q + 2]), __uint_as_float(w[4 * q + 3]));
                            }
                            if (sp == 0) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] = w[i];
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(w[i]));
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ptx::st_shared_v4(row_addr + (static_cast<uint32_t>((hh * 4 + q) ^ (lane & 7)) << 4),
                                              v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    }
                }
            }
        }
        ptx::fence_proxy_async_smem();             // the staging is the source of bulk copies
        // ---- exchange: each warp pushes the boxes it staged to their owners
        // (a box of 32 rows x 32 columns is 256 pieces; a rank's share is a
        // whole number of boxes), so the copies start while other warps stage
        if (Q > 1) {
            ptx::cluster_wait();                   // every peer's receive barrier is set up
            __syncwarp();
            if (lane == 0) {
                for (int jb = half * (BN / 64); jb < (half + 1) * (BN / 64); ++jb) {
                    const int b = jb * 4 + quarter;
                    const int r = (b * 256) / share;
                    if (r == rank) continue;
                    const uint32_t slot = static_cast<uint32_t>(rank - (rank > r ? 1 : 0));
                    ptx::bulk_copy_to_cluster(ptx::mapa(recv + (slot * static_cast<uint32_t>(share) +
                                                                 static_cast<uint32_t>(b * 256 - r * share)) * 16u, r),
                                              E + static_cast<uint32_t>(b) * 4096u, 4096u, ptx::mapa(recv_bar, r));
                }
            }
        }
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (warp == 1 && h == kHalves - 1) {
            // after a time-out the MMAs may still run: wait for them (normal
            // limit) before freeing their tensor memory.  `aborted` is the
            // same in every thread (acc_ok is per thread), and the warp
            // reconverges before the warp-wide deallocation.
            if (aborted) ptx::mbar_wait_bounded(acc_bar, 0, args.wait_limit_ns);
            __syncwarp();
            ptx::tc_fence_after_sync();
            ptx::tmem_dealloc(tmem, Sh::kTmemCols * static_cast<uint32_t>(cpc));
        }
        if (!ptx::mbar_wait_bounded(recv_bar, 0, args.wait_limit_ns) && tid == 0) atomicOr(&g_device_status, 16u);
        if (Q > 1) ptx::cluster_arrive_relaxed();  // everything bound for this CTA has landed

        // ---- epilogue 2: sums of each owned piece over the cluster's ranks.
        // Eight warps do this part, so it is bound by latency, not bandwidth: the
        // shared-memory base of every rank's contribution is computed once, and
        // each thread loads both of its pieces (2 x Q float4) before it adds and
        // stores.
        // the first global stores: the previous grid must have finished (it
        // may still read what these overwrite, or write the same outputs),
        // unless no launch in flight reads or writes them (overlap 2)
        if (args.overlap == 1) ptx::grid_dependency_wait();
        const int row0 = m_tile * TM + h * kTileM, col0 = n_tile * BN;
        const size_t MN = static_cast<size_t>(args.M) * args.N;
        const int rows_here = args.M - row0;                               // tile rows below M
        const size_t tile0 = static_cast<size_t>(row0) * args.N + col0;   // the tile's first element
        uint32_t rbase[Q];   // plus a piece's staging offset: that rank's contribution to the piece
        const uint32_t slot_bytes = static_cast<uint32_t>(share) * 16u;
#pragma unroll
        for (int r = 0; r < Q; ++r)
            rbase[r] = r == rank ? E
                                 : recv + static_cast<uint32_t>(r - (r > rank ? 1 : 0)) * slot_bytes -
                                       static_cast<uint32_t>(my_lo) * 16u;
        auto gather = [&](const Piece &p, float4 (&v)[Q]) {
#pragma unroll
            for (int r = 0; r < Q; ++r) v[r] = ptx::ld_shared_v4(rbase[r] + p.off);
        };
        auto tile_elem = [&](const Piece &p) { return tile0 + static_cast<size_t>(p.row) * args.N + p.col; };
        // the chunk sum of one split (Q == CC): the chunks in pairs
        auto chunk_sum = [&](const float4 (&v)[Q]) { return pair_sum<Q>(v); };
        if (args.split_sum != 2) {
            float *const Ps = P + static_cast<size_t>(s) * MN;
            for (int g0 = my_lo + tid; g0 < my_hi; g0 += 2 * kThreads) {
                const int g1 = g0 + kThreads;
                const Piece p0 = piece_at(g0), p1 = piece_at(min(g1, my_hi - 1));
                float4 v0[Q], v1[Q];
                gather(p0, v0);
                gather(p1, v1);
                const float4 a0 = chunk_sum(v0), a1 = chunk_sum(v1);
                if (p0.row < rows_here) *reinterpret_cast<float4 *>(Ps + tile_elem(p0)) = a0;
                if (g1 < my_hi && p1.row < rows_here) *reinterpret_cast<float4 *>(Ps + tile_elem(p1)) = a1;
            }
        } else if (P != nullptr && !whole_k) {   // (whole_k: the partials were stored while staging)
            cluster_split_sum_for<Q, true>(CC, rbase, my_lo + tid, my_hi, rows_here, tile0, args.N, MN, P, out);
        } else {
            cluster_split_sum_for<Q, false>(CC, rbase, my_lo + tid, my_hi, rows_here, tile0, args.N, MN, nullptr,
                                            out);
        }
    }
    // overlap 2 stored without waiting: the grid still finishes after the
    // previous one, so that grids finish in launch order.  One CTA waiting
    // is enough for that; the others leave at once and free their SM for
    // the next launches.
    if (args.overlap == 2 && blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 &&
        blockIdx.z == gridDim.z - 1)
        ptx::grid_dependency_wait();
    if (Q > 1) ptx::cluster_wait();            // no CTA leaves while its staging may still be copied from
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
// Element type of an operand: 0 F16, 1 BF16, 2 F32.
CUtensorMapDataType map_type(int et)
{
    return et == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                   : et == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}
int elem_of(int et) { return et == 2 ? 4 : 2; }

// A tensor map depends only on the arguments that encode it (address, shape,
// box, element type), not on the data, so calls that repeat them reuse it:
// each host thread keeps the last kMapCache maps it encoded.
struct MapKey {
    const void *ptr;
    int64_t rows, K;
    int box_rows, kbs, et, rank;
    bool operator==(const MapKey &o) const
    {
        return ptr == o.ptr && rows == o.rows && K == o.K && box_rows == o.box_rows && kbs == o.kbs &&
               et == o.et && rank == o.rank;
    }
};
constexpr int kMapCache = 16;
struct MapEntry {
    CUtensorMap map;
    MapKey key;
    bool valid;
};
thread_local MapEntry t_maps[kMapCache];
thread_local int t_map_next = 0;

template <typename Encode>
bool cached_map(CUtensorMap *map, const MapKey &key, Encode encode)
{
    for (const MapEntry &e : t_maps)
        if (e.valid && e.key == key) {
            *map = e.map;
            return true;
        }
    if (!encode(map)) return false;
    MapEntry &slot = t_maps[t_map_next];
    slot.map = *map;
    slot.key = key;
    slot.valid = true;
    t_map_next = (t_map_next + 1) % kMapCache;
    return true;
}

// Row-major [rows, K] matrix, box = box_rows x one 128-byte row (64 16-bit
// or 32 F32 elements), 128-byte swizzle.
bool encode_operand_uncached(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows, int et)
{
    auto fn = encode_fn();
    if (!fn) {
        note_message("cuTensorMapEncodeTiled is not available from the driver", 0);
        return false;
    }
    const int e = elem_of(et);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * e};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / e), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, map_type(et), 2,
                    const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) note_message("cuTensorMapEncodeTiled failed", static_cast<int>(r));
    return r == CUDA_SUCCESS;
}

bool encode_operand(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows, int et)
{
    return cached_map(map, MapKey{ptr, rows, K, box_rows, 1, et, 2},
                      [&](CUtensorMap *m) { return encode_operand_uncached(m, ptr, rows, K, box_rows, et); });
}

// Row-major [rows, K] matrix seen as 3-D (element within a k-block of one
// 128-byte row, row, k-block), box = k-block x box_rows x kbs, 128-byte
// swizzle: one load brings kbs k-blocks of a tile.  Needs K to be a whole
// number of k-blocks, so that no k-block runs past the end of a row.
bool encode_operand_3d_uncached(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows, int kbs,
                                int et)
{
    auto fn = encode_fn();
    if (!fn) {
        note_message("cuTensorMapEncodeTiled is not available from the driver", 0);
        return false;
    }
    const int e = elem_of(et), kb = 128 / e;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kb), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(K / kb)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * e, 128};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kb), static_cast<cuuint32_t>(box_rows),
                         static_cast<cuuint32_t>(kbs)};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, map_type(et), 3,
                          const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) note_message("cuTensorMapEncodeTiled (3-D) failed", static_cast<int>(r));
    return r == CUDA_SUCCESS;
}

bool encode_operand_3d(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows, int kbs, int et)
{
    return cached_map(map, MapKey{ptr, rows, K, box_rows, kbs, et, 3},
                      [&](CUtensorMap *m) { return encode_operand_3d_uncached(m, ptr, rows, K, box_rows, kbs, et); });
}

// Opts the kernel into the device's full dynamic shared memory (what is left
// of the per-block opt-in limit after its static shared memory); once per
// device.
template <int BN, int Q, bool KN, bool X3, int TM, int G>
cudaError_t prepare_kernel_attrs()
{
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return note_error(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return note_error(e, "cudaDeviceGetAttribute(MaxSharedMemoryPerBlockOptin)");
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, tc_splitk_kernel<BN, Q, KN, X3, TM, G>);
    if (e != cudaSuccess) return note_error(e, "cudaFuncGetAttributes(tc_splitk_kernel)");
    const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
    e = cudaFuncSetAttribute(tc_splitk_kernel<BN, Q, KN, X3, TM, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dyn);
    if (e != cudaSuccess) return note_error(e, "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)");
    if (dev >= 0 && dev < 64) done[dev] = true;
    return cudaSuccess;
}

template <int BN, int Q, bool KN, bool X3, int TM = kTileM, int G = 1>
cudaError_t launch_bn(const TcOperands<G> &ops, const TcArgs &args, const TilePlan &plan, cudaStream_t stream)
{
    cudaError_t e = prepare_kernel_attrs<BN, Q, KN, X3, TM, G>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = plan.grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
    if (plan.cluster > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = 1;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = plan.cluster;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return note_error(cudaLaunchKernelEx(&cfg, tc_splitk_kernel<BN, Q, KN, X3, TM, G>, ops, args),
                      "cudaLaunchKernelEx(tc_splitk_kernel)");
}

template <int BN, bool KN, bool X3, int G = 1>
cudaError_t launch_cluster(const TcOperands<G> &ops, const TcArgs &args, const TilePlan &plan, cudaStream_t stream)
{
    switch (plan.cluster) {
    case 1: return launch_bn<BN, 1, KN, X3, kTileM, G>(ops, args, plan, stream);
    case 2: return launch_bn<BN, 2, KN, X3, kTileM, G>(ops, args, plan, stream);
    case 4: return launch_bn<BN, 4, KN, X3, kTileM, G>(ops, args, plan, stream);
    case 8: return launch_bn<BN, 8, KN, X3, kTileM, G>(ops, args, plan, stream);
    default: return note_error(cudaErrorInvalidConfiguration, "cluster size");
    }
}

}  // namespace


namespace {

int elem_code(const GemmProblem &pr) { return pr.f32 ? 2 : pr.bf16 ? 1 : 0; }

// The TMA maps of one problem's A and B for a plan.
bool encode_problem(const GemmProblem &pr, const TilePlan &plan, CUtensorMap *ta, CUtensorMap *tb)
{
    const int et = elem_code(pr);
    const int kbs = plan.three_d ? plan.kbs : 1;
    const bool ok_a = plan.three_d ? encode_operand_3d(ta, pr.A, pr.M, pr.K, plan.tile_m, plan.kbs, et)
                                   : encode_operand(ta, pr.A, pr.M, pr.K, plan.tile_m, et);
    // the [K,N] weight is a row-major matrix of K rows of N: boxes of 64
    // columns by kbs*64 rows
    const bool ok_b = pr.b_kn ? encode_operand(tb, pr.B, pr.K, pr.N, kbs * kBlockK, et)
                              : plan.three_d ? encode_operand_3d(tb, pr.B, pr.N, pr.K, plan.bn, plan.kbs, et)
                                             : encode_operand(tb, pr.B, pr.N, pr.K, plan.bn, et);
    return ok_a && ok_b;
}

template <int G>
void set_problem(TcOperands<G> &ops, int g, const GemmProblem &pr, const TilePlan &plan)
{
    ops.P[g] = pr.P;
    ops.out[g] = plan.fused ? pr.out : nullptr;
    ops.A[g] = static_cast<const uint8_t *>(pr.A);
    ops.B[g] = static_cast<const uint8_t *>(pr.B);
}

TcArgs make_args(const GemmProblem &pr, const TilePlan &plan)
{
    const int et = elem_code(pr);
    TcArgs a = {};
    a.split_sum = plan.split_sum;
    a.M = static_cast<int>(pr.M);
    a.N = static_cast<int>(pr.N);
    a.K = static_cast<int>(pr.K);
    a.S = static_cast<int>(pr.S);
    a.kps = static_cast<int>(pr.kps);
    a.group = 1;
    a.m_tiles = static_cast<int>((pr.M + plan.tile_m - 1) / plan.tile_m);
    a.chunks = plan.chunks;
    a.chunk_len = plan.chunk_len;
    a.stages = plan.stages;
    a.kbs = plan.kbs;
    a.three_d = plan.three_d;
    a.share = plan.share;
    a.region0 = plan.region0;
    a.bf16 = pr.bf16 ? 1 : 0;
    a.wait_limit_ns = kWaitLimitNs;
    a.acc_probe = pr.acc_probe ? 1 : 0;
    a.a_bytes = static_cast<uint64_t>(pr.M * pr.K) * elem_of(et);
    a.b_bytes = static_cast<uint64_t>(pr.N * pr.K) * elem_of(et);
    // a launch that starts beside the previous one loads its own operands at
    // once; prefetching them into L2 only adds requests
    a.prefetchers = pr.overlap ? 0 : plan.prefetchers;
    a.rows_first = plan.rows_first;
    a.overlap = pr.overlap ? (pr.store_early ? 2 : 1) : 0;
    a.recv_in_ring = plan.recv_in_ring && plan.cluster > 1 ? 1 : 0;
    a.cpc = plan.cpc;
    return a;
}

}  // namespace

namespace {

// The plan and problem checks every launch makes before encoding anything.
cudaError_t check_plan(const GemmProblem &pr, const TilePlan &plan)
{
    const bool chunks_ok = (plan.chunks & (plan.chunks - 1)) == 0 && plan.chunks >= 1 && plan.chunks <= kMaxChunks &&
                           (plan.cluster * plan.cpc) % plan.chunks == 0;
    // several chunks per CTA: each its own accumulator (at most 128 tensor-
    // memory columns in all), its chunks whole k-blocks of whole stages
    // (or every chunk of every split: full splits that the chunks tile, no cluster)
    const bool whole_k = plan.cpc > plan.chunks;
    const int kbe = plan.x3 ? 32 : kBlockK;   // elements of a k-block
    const bool pair = plan.cpc == 2 && plan.chunks % 2 == 0;
    const bool whole = whole_k && !plan.x3 && plan.cpc == pr.S * plan.chunks && plan.cluster == 1 &&
                       pr.K == pr.S * pr.kps && pr.kps == static_cast<int64_t>(plan.chunks) * plan.chunk_len;
    const bool cpc_ok = plan.cpc == 1 ||
                        ((pair || whole) && plan.tile_m == kTileM && tmem_fits(plan.bn * plan.cpc, plan.smem_bytes) &&
                         plan.chunk_len % kbe == 0 && (plan.chunk_len / kbe) % plan.kbs == 0 &&
                         static_cast<int64_t>(plan.grid.z) * plan.cpc == pr.S * plan.chunks);
    if (!cpc_ok) return note_error(cudaErrorInvalidConfiguration, "chunks per CTA out of range");
    if (plan.cluster > kMaxChunks || plan.stages > kMaxStages || plan.kbs < 1 || plan.kbs > kMaxKbs ||
        plan.smem_bytes > kSmemLimit || !chunks_ok)
        return note_error(cudaErrorInvalidConfiguration, "tile plan out of range");
    if (plan.fused && (pr.out == nullptr || plan.split_sum != 2))
        return note_error(cudaErrorInvalidValue, "fused launch without output or cluster split sum");
    if (pr.P == nullptr && plan.split_sum != 2)
        return note_error(cudaErrorInvalidValue, "partials are needed unless the cluster sums the splits");
    if (pr.f32 && (pr.b_kn || !plan.x3))
        return note_error(cudaErrorInvalidValue, "F32 operands need a 3xTF32 plan and the [N,K] weight");
    const bool tile_m_ok = plan.tile_m == kTileM || (plan.tile_m == 2 * kTileM && plan.bn == 256 &&
                                                     plan.cluster == 1 && !plan.x3);
    if (!tile_m_ok) return note_error(cudaErrorInvalidConfiguration, "256-row tile plan out of range");
    if (plan.recv_in_ring && static_cast<size_t>(kTileM) * plan.bn * 4 +
                                 static_cast<size_t>(plan.cluster - 1) * plan.share * 16 >
                             plan.region0)
        return note_error(cudaErrorInvalidConfiguration, "receive slots outside the stage ring");
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_tc(const GemmProblem &pr, const TilePlan &plan, cudaStream_t stream)
{
    const cudaError_t ce = check_plan(pr, plan);
    if (ce != cudaSuccess) return ce;
    TcOperands<1> ops = {};
    if (!encode_problem(pr, plan, &ops.tm[0][0], &ops.tm[0][1])) return cudaErrorInvalidValue;
    set_problem(ops, 0, pr, plan);
    const TcArgs a = make_args(pr, plan);
    // operand variants: [N,K] weight, [K,N] weight, F32 as 3xTF32
    const int variant = pr.f32 ? 2 : pr.b_kn ? 1 : 0;
    if (plan.tile_m == 2 * kTileM)
        return variant == 1 ? launch_bn<256, 1, true, false, 2 * kTileM>(ops, a, plan, stream)
                            : launch_bn<256, 1, false, false, 2 * kTileM>(ops, a, plan, stream);
    switch (plan.bn * 4 + variant) {
    case 64 * 4 + 0: return launch_cluster<64, false, false>(ops, a, plan, stream);
    case 64 * 4 + 1: return launch_cluster<64, true, false>(ops, a, plan, stream);
    case 64 * 4 + 2: return launch_cluster<64, false, true>(ops, a, plan, stream);
    case 128 * 4 + 0: return launch_cluster<128, false, false>(ops, a, plan, stream);
    case 128 * 4 + 1: return launch_cluster<128, true, false>(ops, a, plan, stream);
    case 128 * 4 + 2: return launch_cluster<128, false, true>(ops, a, plan, stream);
    case 256 * 4 + 0: return launch_cluster<256, false, false>(ops, a, plan, stream);
    case 256 * 4 + 1: return launch_cluster<256, true, false>(ops, a, plan, stream);
    case 256 * 4 + 2: return launch_cluster<256, false, true>(ops, a, plan, stream);
    default: return note_error(cudaErrorInvalidConfiguration, "tile width");
    }
}

// ---- grouping consecutive independent calls into one launch (graph capture)
//
// Inside a capture, a call that may store before the launch before it ends
// (splitk_chain.cu: nothing in flight reads or writes its operands or outputs)
// and that has the same shape and plan as that launch joins it: the launch's
// kernel node gets the call's operands as one more problem (the group index
// is the high part of blockIdx.y) and a grid that covers it, and no node is
// added.  The problems of a group are independent, so their CTAs may run in
// any order; the node keeps its place in the chain.  A group holds at most
// kMaxGroup problems; grouped launches use the kernel instantiated for
// kMaxGroup problems (16-bit operands, 128-row tiles, BN <= 128).
namespace {

struct GroupState {
    bool valid = false;
    unsigned long long capture = 0;
    cudaGraphNode_t node = nullptr;
    uint64_t stamp = 0;
    // what every problem of the group shares
    int64_t M = 0, N = 0, K = 0, S = 0, kps = 0;
    bool bf16 = false, b_kn = false, keep_p = false, overlap = false, store_early = false;
    TilePlan plan = {};
    // the node's launch
    void *func = nullptr;
    size_t smem = 0;
    TcOperands<kMaxGroup> ops = {};
    TcArgs args = {};
    int n = 0;
    GemmProblem head = {};   // the first problem, as launched
};

constexpr int kGroupSlots = 16;
std::mutex g_group_mu;
GroupState g_groups[kGroupSlots];
uint64_t g_group_clock = 0;

bool same_plan(const TilePlan &a, const TilePlan &b)
{
    return a.bn == b.bn && a.chunks == b.chunks && a.chunk_len == b.chunk_len && a.stages == b.stages &&
           a.kbs == b.kbs && a.three_d == b.three_d && a.cluster == b.cluster && a.fused == b.fused &&
           a.split_sum == b.split_sum && a.share == b.share && a.region0 == b.region0 && a.x3 == b.x3 &&
           a.rows_first == b.rows_first && a.tile_m == b.tile_m && a.compact == b.compact &&
           a.recv_in_ring == b.recv_in_ring && a.cpc == b.cpc && a.grid.x == b.grid.x && a.grid.y == b.grid.y &&
           a.grid.z == b.grid.z && a.smem_bytes == b.smem_bytes;
}

}  // namespace

// A launch heads a group with any tensor-core plan (16-bit operands, or F32
// with the [N,K] weight) of tiles 128 rows by at most 128 columns in column
// order (the grouped kernels' instances); later calls join it only with the
// same compact plan, or convert it (convert_head).
bool head_groupable(const GemmProblem &pr, const TilePlan &plan)
{
    return plan.x3 == pr.f32 && !(pr.f32 && pr.b_kn) && !pr.acc_probe && plan.tile_m == kTileM && plan.bn <= 128 &&
           !plan.rows_first;
}

namespace {

bool groupable(const GemmProblem &pr, const TilePlan &plan)
{
    return plan.compact && head_groupable(pr, plan);
}

// The grouped kernel of a plan: one instance per tile width (64, 128),
// operand form (16-bit [N,K] or [K,N], F32 [N,K]) and cluster size.  `op`
// asks for its function, its shared-memory attribute, or a launch.
enum class GroupedOp { kFunc, kPrepare, kLaunch };

template <int BN, int Q, bool KN, bool X3>
cudaError_t grouped_op_q(GroupedOp op, void **func, const TcOperands<kMaxGroup> *ops, const TcArgs *a,
                         const TilePlan *plan, cudaStream_t stream)
{
    switch (op) {
    case GroupedOp::kFunc:
        *func = reinterpret_cast<void *>(tc_splitk_kernel<BN, Q, KN, X3, kTileM, kMaxGroup>);
        return cudaSuccess;
    case GroupedOp::kPrepare: return prepare_kernel_attrs<BN, Q, KN, X3, kTileM, kMaxGroup>();
    default: return launch_bn<BN, Q, KN, X3, kTileM, kMaxGroup>(*ops, *a, *plan, stream);
    }
}

template <int BN, bool KN, bool X3>
cudaError_t grouped_op_bn(GroupedOp op, int q, void **func, const TcOperands<kMaxGroup> *ops, const TcArgs *a,
                          const TilePlan *plan, cudaStream_t stream)
{
    switch (q) {
    case 1: return grouped_op_q<BN, 1, KN, X3>(op, func, ops, a, plan, stream);
    case 2: return grouped_op_q<BN, 2, KN, X3>(op, func, ops, a, plan, stream);
    case 4: return grouped_op_q<BN, 4, KN, X3>(op, func, ops, a, plan, stream);
    case 8: return grouped_op_q<BN, 8, KN, X3>(op, func, ops, a, plan, stream);
    default: return note_error(cudaErrorInvalidConfiguration, "cluster size");
    }
}

cudaError_t grouped_op(GroupedOp op, const TilePlan &plan, bool kn, void **func,
                       const TcOperands<kMaxGroup> *ops = nullptr, const TcArgs *a = nullptr,
                       cudaStream_t stream = nullptr)
{
    const int q = plan.cluster;
    switch (plan.bn * 4 + (kn ? 2 : 0) + (plan.x3 ? 1 : 0)) {
    case 64 * 4 + 0: return grouped_op_bn<64, false, false>(op, q, func, ops, a, &plan, stream);
    case 64 * 4 + 2: return grouped_op_bn<64, true, false>(op, q, func, ops, a, &plan, stream);
    case 64 * 4 + 1: return grouped_op_bn<64, false, true>(op, q, func, ops, a, &plan, stream);
    case 128 * 4 + 0: return grouped_op_bn<128, false, false>(op, q, func, ops, a, &plan, stream);
    case 128 * 4 + 2: return grouped_op_bn<128, true, false>(op, q, func, ops, a, &plan, stream);
    case 128 * 4 + 1: return grouped_op_bn<128, false, true>(op, q, func, ops, a, &plan, stream);
    default: return note_error(cudaErrorInvalidConfiguration, "tile width or operand form");
    }
}

}  // namespace

cudaError_t launch_tc_grouped(const GemmProblem &pr, const TilePlan &plan, cudaStream_t stream,
                              unsigned long long capture)
{
    if (!head_groupable(pr, plan) || capture == 0) return launch_tc(pr, plan, stream);
    cudaError_t e = check_plan(pr, plan);
    if (e != cudaSuccess) return e;
    GroupState st;
    if (!encode_problem(pr, plan, &st.ops.tm[0][0], &st.ops.tm[0][1])) return cudaErrorInvalidValue;
    set_problem(st.ops, 0, pr, plan);
    st.args = make_args(pr, plan);
    st.args.group = 1;
    e = grouped_op(GroupedOp::kLaunch, plan, pr.b_kn, nullptr, &st.ops, &st.args, stream);
    if (e != cudaSuccess) return e;
    if (grouped_op(GroupedOp::kFunc, plan, pr.b_kn, &st.func) != cudaSuccess) st.func = nullptr;
    // the node just captured, which later calls may join
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    unsigned long long id = 0;
    const cudaGraphNode_t *deps = nullptr;
    size_t nd = 0;
    if (cudaStreamGetCaptureInfo(stream, &cs, &id, nullptr, &deps, nullptr, &nd) != cudaSuccess ||
        cs != cudaStreamCaptureStatusActive || id != capture || nd != 1 || st.func == nullptr)
        return cudaSuccess;   // launched; just not joinable
    st.valid = true;
    st.capture = capture;
    st.node = deps[0];
    st.M = pr.M; st.N = pr.N; st.K = pr.K; st.S = pr.S; st.kps = pr.kps;
    st.bf16 = pr.bf16; st.b_kn = pr.b_kn; st.keep_p = pr.P != nullptr;
    st.overlap = pr.overlap; st.store_early = pr.store_early;
    st.plan = plan;
    st.smem = plan.smem_bytes;
    st.n = 1;
    st.head = pr;
    std::lock_guard<std::mutex> lock(g_group_mu);
    // the capture's slot, else a free one, else the least recently used
    GroupState *slot = nullptr;
    for (GroupState &g : g_groups)
        if (g.valid && g.capture == capture) slot = &g;
    if (!slot)
        for (GroupState &g : g_groups)
            if (!g.valid) {
                slot = &g;
                break;
            }
    if (!slot) {
        slot = &g_groups[0];
        for (GroupState &g : g_groups)
            if (g.stamp < slot->stamp) slot = &g;
    }
    st.stamp = ++g_group_clock;
    *slot = st;
    return cudaSuccess;
}

cudaError_t launch_tc_batch(const GemmProblem *prs, int n, const TilePlan &plan, cudaStream_t stream)
{
    if (n < 1 || n > kMaxGroup || !groupable(prs[0], plan)) return cudaErrorInvalidValue;
    TcOperands<kMaxGroup> ops = {};
    for (int i = 0; i < n; ++i) {
        const cudaError_t e = check_plan(prs[i], plan);
        if (e != cudaSuccess) return e;
        if (!encode_problem(prs[i], plan, &ops.tm[i][0], &ops.tm[i][1])) return cudaErrorInvalidValue;
        set_problem(ops, i, prs[i], plan);
    }
    TcArgs a = make_args(prs[0], plan);
    a.group = n;
    a.prefetchers = 0;
    TilePlan bp = plan;
    bp.grid.y *= static_cast<unsigned>(n);   // blockIdx.y = problem * row tiles + row tile
    bp.prefetchers = 0;
    return grouped_op(GroupedOp::kLaunch, bp, prs[0].b_kn, nullptr, &ops, &a, stream);
}

namespace {

// The first launch of a run takes its usual (eager) plan, which alone in a
// graph runs fastest.  The first call after it with the same shape converts
// that launch to its own plan (compact, or whole-K blocks) and joins it: the
// node gets that plan's kernel, cluster size, grid and shared memory and both
// problems.  Where a step fails the node is left as it was (its cluster
// attribute restored) and the call launches on its own; should the restore
// itself fail, *broken tells the caller, whose call then fails.
bool convert_head(GroupState &st, const GemmProblem &pr, const TilePlan &plan, bool *broken)
{
    if (st.n != 1 || !groupable(pr, plan)) return false;
    const GemmProblem &h = st.head;
    if ((h.out != nullptr) != (plan.split_sum == 2) || (pr.out != nullptr) != (plan.split_sum == 2)) return false;
    if (check_plan(h, plan) != cudaSuccess) return false;
    TcOperands<kMaxGroup> ops = {};
    if (!encode_problem(h, plan, &ops.tm[0][0], &ops.tm[0][1]) ||
        !encode_problem(pr, plan, &ops.tm[1][0], &ops.tm[1][1]))
        return false;
    set_problem(ops, 0, h, plan);
    set_problem(ops, 1, pr, plan);
    TcArgs a = make_args(h, plan);   // the head's overlap mode
    a.group = 2;
    a.prefetchers = 0;
    void *func = nullptr;
    if (grouped_op(GroupedOp::kFunc, plan, h.b_kn, &func) != cudaSuccess ||
        grouped_op(GroupedOp::kPrepare, plan, h.b_kn, nullptr) != cudaSuccess || func == nullptr)
        return false;
    // The cluster size first: the new size divides the launch's current grid
    // (a cluster holds the splits and chunks of a tile, fewer of them once
    // merged), so the node is valid in between; the new parameters then.
    cudaLaunchAttributeValue old = {}, one = {};
    if (cudaGraphKernelNodeGetAttribute(st.node, cudaLaunchAttributeClusterDimension, &old) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    one.clusterDim.x = one.clusterDim.y = 1;
    one.clusterDim.z = static_cast<unsigned>(plan.cluster);
    if (cudaGraphKernelNodeSetAttribute(st.node, cudaLaunchAttributeClusterDimension, &one) != cudaSuccess) {
        (void)cudaGetLastError();   // the node is as it was
        return false;
    }
    cudaKernelNodeParams kp = {};
    kp.func = func;
    kp.gridDim = dim3(plan.grid.x, plan.grid.y * 2u, plan.grid.z);
    kp.blockDim = dim3(kThreads, 1, 1);
    kp.sharedMemBytes = static_cast<unsigned>(plan.smem_bytes);
    void *params[2] = {&ops, &a};
    kp.kernelParams = params;
    kp.extra = nullptr;
    if (cudaGraphKernelNodeSetParams(st.node, &kp) != cudaSuccess) {
        (void)cudaGetLastError();
        st.valid = false;
        if (cudaGraphKernelNodeSetAttribute(st.node, cudaLaunchAttributeClusterDimension, &old) != cudaSuccess) {
            (void)cudaGetLastError();
            *broken = true;   // old kernel, new cluster size: the capture must not be used
            note_error(cudaErrorUnknown, "grouped launch: graph node left with a mismatched cluster size");
        }
        return false;
    }
    st.plan = plan;
    st.func = func;
    st.smem = plan.smem_bytes;
    st.ops = ops;
    st.args = a;
    st.n = 2;
    return true;
}

}  // namespace

bool join_group(const GemmProblem &pr, const TilePlan &plan, unsigned long long capture, cudaGraphNode_t dep,
                int *group_size, int *mode, bool *broken)
{
    *broken = false;
    if (!groupable(pr, plan) || capture == 0 || dep == nullptr) return false;
    if (check_plan(pr, plan) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_group_mu);
    GroupState *st = nullptr;
    for (GroupState &g : g_groups)
        if (g.valid && g.capture == capture) st = &g;
    if (!st || st->node != dep || st->n >= kMaxGroup) return false;
    const bool same_shape = st->M == pr.M && st->N == pr.N && st->K == pr.K && st->S == pr.S &&
                            st->kps == pr.kps && st->bf16 == pr.bf16 && st->b_kn == pr.b_kn &&
                            st->keep_p == (pr.P != nullptr) && (st->head.out != nullptr) == (pr.out != nullptr);
    if (!same_shape) return false;
    if (!same_plan(st->plan, plan)) {
        if (!convert_head(*st, pr, plan, broken)) return false;
        st->stamp = ++g_group_clock;
        if (group_size) *group_size = st->n;
        if (mode) *mode = st->overlap ? (st->store_early ? 2 : 1) : 0;
        return true;
    }
    const int g = st->n;
    if (!encode_problem(pr, plan, &st->ops.tm[g][0], &st->ops.tm[g][1])) return false;
    set_problem(st->ops, g, pr, plan);
    TcArgs a = st->args;
    a.group = g + 1;
    a.prefetchers = 0;   // several problems: no early CTAs prefetch one of them
    cudaKernelNodeParams kp = {};
    kp.func = st->func;
    kp.gridDim = dim3(plan.grid.x, plan.grid.y * static_cast<unsigned>(g + 1), plan.grid.z);
    kp.blockDim = dim3(kThreads, 1, 1);
    kp.sharedMemBytes = static_cast<unsigned>(st->smem);
    void *params[2] = {&st->ops, &a};
    kp.kernelParams = params;
    kp.extra = nullptr;
    if (cudaGraphKernelNodeSetParams(st->node, &kp) != cudaSuccess) {
        (void)cudaGetLastError();
        st->valid = false;   // leave the node as it was; the call launches on its own
        return false;
    }
    st->args = a;
    st->n = g + 1;
    st->stamp = ++g_group_clock;
    if (group_size) *group_size = st->n;
    if (mode) *mode = st->overlap ? (st->store_early ? 2 : 1) : 0;
    return true;
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
    return note_error(cudaGetLastError(), "wait_selftest_kernel launch");
}

}  // namespace splitk
