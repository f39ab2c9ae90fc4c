// splitk_plan.cu -- the tile planner: which tiles, chunks, stages, cluster
// and shared memory a tensor-core launch takes for a shape, and the cost
// model the split-count chooser uses.  Host code only; the kernel and its
// launches are in splitk_tc.cu, which checks every plan again before it
// launches (check_plan).
//
// The operation it plans is the partial pass (and optionally the split sum)
// of the pages "Aligned shared rows for pipelined NAX on CUDA" and "Wider
// consecutive-weight NAX GEMM" (sections "Contract and correctness" /
// "Launch contract and correctness"); the tiling is the library's own.

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "splitk_internal.h"

namespace splitk {

// Tensor-memory columns a CTA may allocate for its shared memory, so that the
// CTAs of these kernels that fit on an SM by shared memory (228 KB, 1 KB of
// it reserved per CTA) always fit in its 512 columns and no allocation waits
// on a CTA that may wait in turn: at most one column per 512 bytes, or 256
// columns from 100 KB on.  Every plan has at least 32 KB per 64 columns (its
// accumulator staging area), so the CTAs beside a 256-column one (at least
// 101 KB with the reserve) hold at most 256 columns more: two 256-column
// CTAs leave no room for a third CTA, one beside a 128-column CTA (66 KB)
// leaves room for at most one of 64 (34 KB), and 64-column CTAs alone keep
// to 2 columns per KB.
constexpr size_t kTmem256Smem = 100 * 1024;
bool tmem_fits(int cols, size_t smem)
{
    return static_cast<size_t>(cols) * 512 <= smem || (cols == 256 && smem >= kTmem256Smem) ||
           (cols == 512 && smem >= kSmemLimit);   // all of a block's shared memory: alone on its SM
}

namespace {

int g_override_bn = 0, g_override_chunks = 0, g_override_kbs = 0;

// One k-block is one 128-byte row of every operand row (tm rows of A, bn of
// B); a 3xTF32 stage holds the lo parts too.
size_t stage_bytes(int bn, int kbs, bool x3 = false, int tm = kTileM)
{
    return static_cast<size_t>(tm + bn) * 128 * kbs * (x3 ? 2 : 1);
}
size_t epi_bytes(int bn) { return static_cast<size_t>(kTileM) * bn * 4; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
// The compact layout: two or three CTAs to an SM (228 KB of shared memory,
// 1 KB of it reserved per CTA, plus the kernel's static barriers), so that
// the next operations' CTAs can start beside this one's.
constexpr size_t kCompactSmemLimit = 112 * 1024;
constexpr size_t kCompact3SmemLimit = 74 * 1024;

// Dynamic shared memory of a plan: the stage ring (or the accumulator
// staging, if larger), one receive slot per peer, and 1 KB of alignment slack.
// With the receive slots in the ring (rir) they follow the staging area
// inside it, so the ring only has to be at least that large.
size_t smem_for(int bn, int kbs, int stages, int chunks, int share, bool x3 = false, int tm = kTileM,
                bool rir = false)
{
    const size_t recv = static_cast<size_t>(chunks - 1) * share * 16;
    if (rir) return round_up(std::max(stages * stage_bytes(bn, kbs, x3, tm), epi_bytes(bn) + recv), 1024) + 1024;
    const size_t region0 = round_up(std::max(stages * stage_bytes(bn, kbs, x3, tm), epi_bytes(bn)), 1024);
    return region0 + recv + 1024;
}


}  // namespace

void set_tile_override(int bn, int chunks, int kbs)
{
    g_override_bn = bn;
    g_override_chunks = chunks;
    g_override_kbs = kbs;
}

namespace {

// Clusters of q CTAs (one per SM) a GB300 keeps resident at once, from
// cudaOccupancyMaxActiveClusters: 36 of 4, 15 of 8; pairs and single CTAs are
// limited by the SM count.
int resident_clusters(int q)
{
    switch (q) {
    case 1: return 148;
    case 2: return 72;
    case 4: return 36;
    default: return 15;
    }
}

struct StageChoice {
    int kbs = 1, stages = 1;
    bool ok = false;
};

// The largest stage (k-blocks per box) that keeps a chunk's loads double-
// buffered, or all in flight, within `limit` bytes of shared memory, for a
// cluster of q.
StageChoice pick_stages(int bn, int nkb, bool can3d, int q, int share, bool x3 = false, int tm = kTileM,
                        size_t limit = kSmemLimit, bool rir = false, int max_kbs = kMaxKbs)
{
    StageChoice r;
    for (int cand : {kMaxKbs, 2, 1}) {
        if ((!can3d && cand > 1) || cand > max_kbs) continue;
        if (g_override_kbs && cand != std::min(g_override_kbs, can3d ? kMaxKbs : 1)) continue;
        const int want = (nkb + cand - 1) / cand;
        int st = std::min(want, kMaxStages);
        while (st > 1 && smem_for(bn, cand, st, q, share, x3, tm, rir) > limit) --st;
        if (smem_for(bn, cand, st, q, share, x3, tm, rir) > limit) continue;
        if (st < std::min(want, 2) && !g_override_kbs) continue;
        r.kbs = std::min(cand, std::max(nkb, 1));
        r.stages = st;
        r.ok = true;
        return r;
    }
    return r;
}

int share_for(int bn, int q)
{
    const int pieces = kTileM * bn / 4;
    return static_cast<int>(round_up((pieces + q - 1) / q, 8));
}

// Time model of one launch (microseconds), from measurements on GB300: the
// loads are bound by the L2 (about 10.5 TB/s for all SMs) or by one SM's TMA
// intake (about 100 GB/s); staging the accumulator and the owners' stores to
// L2 run near 100 GB/s, the distributed-shared-memory exchange near 30 GB/s
// per SM.
double model_us(int64_t M, int64_t N, int64_t S, int bn, int chunks, int64_t chunk_len, int q, int elem = 2)
{
    const int64_t mt = (M + kTileM - 1) / kTileM;
    const int64_t ctas = mt * (N / bn) * S * chunks;
    const double load = static_cast<double>(kTileM + bn) * chunk_len * elem;  // bytes per CTA
    const double acc = static_cast<double>(kTileM) * bn * 4;
    const double t_load = std::max(load / 1.0e5, ctas * load / 1.05e7);
    const double t_stage = acc / 1.0e5;
    const double t_exchange = acc * (q - 1) / q / 3.0e4;
    // the owner's stores go to L2 (~100 GB/s per SM); the F32 plans were fitted with 30 GB/s,
    // which stands in there for the converter warps' share of the stage time
    const double t_store = acc / q / (elem == 4 ? 3.0e4 : 1.0e5);
    const int64_t per_wave = q > 1 ? static_cast<int64_t>(resident_clusters(q)) * q : 148;
    const int64_t waves = (ctas + per_wave - 1) / per_wave;
    return static_cast<double>(waves) * (t_load + t_stage + t_exchange + t_store);
}

}  // namespace

// Estimated microseconds per call of one tensor-core launch in a stream of
// such calls inside a graph (where independent calls overlap): the layout a
// graph gives it (compact, and for a fused call that follows another, merged
// chunks or whole-K blocks), each CTA living for its loads (per-CTA TMA
// intake ~99 GB/s), its exchange over distributed shared memory (~7.5 GB/s
// per CTA, contended) and its stores (~77 GB/s), the GPU keeping 148 x (CTAs
// per SM) of them at once -- three, two or one by the compact plan's shared
// memory, otherwise what shared memory allows, at most two -- plus a fixed
// 1.53 us, less 0.17 us per doubling of the cluster.  Fitted on GB300 to 110
// measured candidates (BF16, 12 shapes from M32 N64 K128 to M8192 N8192
// K8192, fused and two kernels, 1 to 16 splits, graphs of the same call):
// median error 6%, at most 1.42x.
double estimate_tc_us(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused, bool x3)
{
    const TilePlan p = plan_tc(M, N, K, S, kps, fused, x3, true, fused);
    const double elem = x3 ? 4.0 : 2.0;
    const double ctas = static_cast<double>(p.grid.x) * p.grid.y * p.grid.z;
    const double acc = static_cast<double>(kTileM) * p.bn * 4;
    const double load = static_cast<double>(p.tile_m + p.bn) * p.chunk_len * p.cpc * elem;   // per CTA
    const double exchange = p.cluster > 1 ? acc * (p.cluster - 1) / p.cluster : 0.0;
    const double store = acc / p.cluster;
    int per_sm;
    if (p.compact)
        per_sm = p.smem_bytes <= kCompact3SmemLimit + 1024 ? 3 : (p.smem_bytes <= kCompactSmemLimit + 1024 ? 2 : 1);
    else
        per_sm = std::max(1, std::min(2, static_cast<int>((228 * 1024) / (p.smem_bytes + 1024 + 256))));
    const double cta_us = load / 9.864e4 + exchange / 7.468e3 + store / 7.665e4;
    return 1.534 - 0.1686 * std::log2(static_cast<double>(p.cluster)) +
           cta_us * ctas / (static_cast<double>(resident_clusters(1)) * per_sm);
}

namespace {

TilePlan plan_tc_uncached(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused, bool x3, bool compact,
                          bool whole_ok);

// The plan depends only on the problem's shape, the element width, `fused`,
// the layout asked for and the tile override, so each host thread keeps the
// last kPlanCache plans.
struct PlanKey {
    int64_t M, N, K, S, kps;
    bool fused, x3, compact, whole_ok;
    int ov_bn, ov_chunks, ov_kbs;
    bool operator==(const PlanKey &o) const
    {
        return M == o.M && N == o.N && K == o.K && S == o.S && kps == o.kps && fused == o.fused && x3 == o.x3 &&
               compact == o.compact && whole_ok == o.whole_ok && ov_bn == o.ov_bn && ov_chunks == o.ov_chunks && ov_kbs == o.ov_kbs;
    }
};
constexpr int kPlanCache = 8;
struct PlanEntry {
    PlanKey key;
    TilePlan plan;
    bool valid;
};
thread_local PlanEntry t_plans[kPlanCache];
thread_local int t_plan_next = 0;

}  // namespace

TilePlan plan_tc(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused, bool x3, bool compact,
                 bool whole_ok)
{
    whole_ok = whole_ok && compact;
    const PlanKey key{M, N, K, S, kps, fused, x3, compact, whole_ok, g_override_bn, g_override_chunks, g_override_kbs};
    for (const PlanEntry &e : t_plans)
        if (e.valid && e.key == key) return e.plan;
    const TilePlan p = plan_tc_uncached(M, N, K, S, kps, fused, x3, compact, whole_ok);
    t_plans[t_plan_next] = PlanEntry{key, p, true};
    t_plan_next = (t_plan_next + 1) % kPlanCache;
    return p;
}

namespace {

TilePlan plan_tc_uncached(int64_t M, int64_t N, int64_t K, int64_t S, int64_t kps, bool fused, bool x3, bool compact,
                          bool whole_ok)
{
    // Stages of several k-blocks load as one 3-D box per operand, which the
    // TMA unit moves much faster than the same bytes in 16 KB boxes; that needs
    // every chunk to start on a k-block boundary (64 elements of 16 bits, or
    // 32 F32, one 128-byte row).
    const int kb_elems = x3 ? 32 : kBlockK;
    const bool can3d = K % kb_elems == 0 && kps % kb_elems == 0;
    const int64_t grain = can3d ? kb_elems : 32;
    const int64_t mt = (M + kTileM - 1) / kTileM;
    // Tile width and chunks per split: the cheapest by the model, with a
    // penalty where the splits of a tile cannot share one resident cluster of
    // a power-of-two size (a fused call then runs the separate reduce).  The
    // choice does not depend on `fused`, so both paths add the same chunks in
    // the same order.
    int best_bn = 0, best_c = 0;
    double best = 1e30;
    for (int bn : {64, 128, 256}) {
        if (N % bn) continue;
        if (g_override_bn && N % g_override_bn == 0 && bn != g_override_bn) continue;
        for (int c : {1, 2, 4, 8}) {
            if (g_override_chunks && c != g_override_chunks) continue;
            int64_t len = (kps + c - 1) / c;
            len = (len + grain - 1) / grain * grain;
            if (!g_override_chunks && c > 1 && (c - 1) * len >= kps) continue;   // an always-empty chunk
            const int nkb = static_cast<int>((len + kb_elems - 1) / kb_elems);
            if (!pick_stages(bn, nkb, can3d, c, share_for(bn, c), x3).ok) continue;
            const int64_t tiles = mt * (N / bn);
            const int64_t sq = S * c;
            // a single CTA per tile needs no cluster: its sum is its own tile
            const bool cluster_sum = sq <= kMaxChunks && (sq & (sq - 1)) == 0 &&
                                     (sq == 1 || tiles <= resident_clusters(static_cast<int>(sq))) &&
                                     pick_stages(bn, nkb, can3d, static_cast<int>(sq),
                                                 share_for(bn, static_cast<int>(sq)), x3).ok;
            const double cost = model_us(M, N, S, bn, c, len, c, x3 ? 4 : 2) + (cluster_sum ? 0.0 : 1.5);
            if (cost < best) {
                best = cost;
                best_bn = bn;
                best_c = c;
            }
        }
    }
    if (best_bn == 0) {   // nothing fits the override: smallest tiles, one chunk
        best_bn = 64;
        best_c = 1;
    }
    const int bn = best_bn, chunks = best_c;
    int64_t chunk_len = (kps + chunks - 1) / chunks;
    chunk_len = (chunk_len + grain - 1) / grain * grain;
    const int nkb = static_cast<int>((chunk_len + kb_elems - 1) / kb_elems);
    const int64_t tiles = mt * (N / bn);
    // A fused launch sums the splits inside its clusters, which must then hold
    // every split and chunk of a tile and all be resident at once; where that
    // fails the plan is not fused (split_sum 0) and gemm_bt runs the reduce.
    int q = chunks, split_sum = 0;
    if (fused) {
        const int sq = static_cast<int>(S) * chunks;
        if (sq <= kMaxChunks && (sq & (sq - 1)) == 0 && (sq == 1 || tiles <= resident_clusters(sq)) &&
            pick_stages(bn, nkb, can3d, sq, share_for(bn, sq), x3).ok) {
            q = sq;
            split_sum = 2;
        }
    }
    const int share = share_for(bn, q);
    // 256-row tiles (two accumulators sharing each B operand) load 64 KB per
    // k-block for twice the products of a 128-row tile's 48 KB.  A launch of
    // many tiles is bound by the rate at which each SM takes in its loads, so
    // a 256-row tile takes ~1.36x as long as a 128-row one (the load bytes'
    // ratio; per wave, GB300 measured 1.37-1.44) and wins where halving the
    // tile count saves more than that in waves of 148 CTAs.  Only for one
    // CTA per tile that keeps or sums its own partials, with BN = 256 and
    // 16-bit operands.
    int tm = kTileM;
    if (!x3 && bn == 256 && q == 1 && mt > 1) {
        const int64_t per_row_tile = (N / bn) * S;
        const double waves1 = std::ceil(static_cast<double>(mt * per_row_tile) / resident_clusters(1));
        const double waves2 = std::ceil(static_cast<double>((mt + 1) / 2 * per_row_tile) / resident_clusters(1));
        if (waves1 > 1.0 && waves2 * 1.36 < waves1 && pick_stages(bn, nkb, can3d, 1, share, x3, 2 * kTileM).ok)
            tm = 2 * kTileM;
    }
    const StageChoice sc = pick_stages(bn, nkb, can3d, q, share, x3, tm);
    TilePlan p = {};
    p.cpc = 1;
    p.tile_m = tm;
    p.bn = bn;
    p.chunks = chunks;
    p.chunk_len = static_cast<int>(chunk_len);
    p.stages = sc.stages;
    p.kbs = can3d ? sc.kbs : 1;
    p.three_d = can3d && p.kbs > 1 ? 1 : 0;
    p.fused = split_sum == 2 ? 1 : 0;
    p.split_sum = split_sum;
    p.cluster = q;
    p.share = share;
    p.x3 = x3 ? 1 : 0;
    p.region0 =
        static_cast<uint32_t>(round_up(std::max(p.stages * stage_bytes(bn, p.kbs, x3, tm), epi_bytes(bn)), 1024));
    // CTAs are dispatched x first.  With x over the column tiles, each wave of
    // a launch of more than one wave sweeps B's whole split slab.  Once that
    // slab is more than a quarter of L2 it no longer stays there from wave to
    // wave; if A's slab is the smaller one, walk the row tiles first instead,
    // so that each wave sweeps A (which then stays in L2) and a band of B.
    // On a GB300, M4096 N8192 K4096 (B slab 64 MB) went from 243.7 to 236.4 us
    // fused, while shapes whose slabs both fit (16 MB and less) ran 2-7%
    // slower in row order.
    const int64_t row_tiles = (M + tm - 1) / tm;
    const int64_t ctas = row_tiles * (N / bn) * S * chunks;
    const int64_t clusters = ctas / q;
    const int64_t b_slab = N * kps * (x3 ? 4 : 2);
    p.rows_first = clusters > resident_clusters(q) && mt * kTileM < N && b_slab > (int64_t(32) << 20) &&
                           N / bn <= 65535 ? 1 : 0;
    const unsigned gx = static_cast<unsigned>(N / bn), gy = static_cast<unsigned>(row_tiles);
    const unsigned gz = static_cast<unsigned>(S * chunks);
    p.grid = p.rows_first ? dim3(gy, gx, gz) : dim3(gx, gy, gz);
    // CTAs of the next launch that fit beside this one (whole clusters): they
    // start early under programmatic dependent launch and do the prefetch
    const int64_t spare = std::max<int64_t>(0, static_cast<int64_t>(resident_clusters(q)) - clusters) * q;
    p.prefetchers = static_cast<int>(std::min(spare, ctas));
    // A 256-row tile's CTA takes all the shared memory a block may have, so
    // that no other CTA of these kernels shares its SM: its two accumulators
    // fill the SM's 512 tensor-memory columns.
    p.smem_bytes = tm == 2 * kTileM ? kSmemLimit : smem_for(bn, p.kbs, p.stages, q, share, x3, tm);
    // The compact layout (asked for where consecutive independent operations
    // may run side by side): the same tiles, chunks and cluster, so the same
    // sums in the same order, with the ring cut to what two CTAs per SM
    // allow and the peers' shares received inside it.  Only for launches of
    // one wave (where the next operation's CTAs would otherwise find no room)
    // and tiles of at most 128 columns (three CTAs' accumulators then fit in
    // an SM's 512 tensor-memory columns).  On GB300, a graph of eight
    // independent BF16 M256 N1024 K2048 operations went from 5.9 to 4.2 us
    // per operation with this layout and the early start; the layout alone,
    // with every launch waiting for the one before, was slower (6.7 us).
    // Launches of more CTAs than half the SMs, with clusters of at most 4
    // (whose kernels keep to 85 registers), cut the ring further, to three
    // CTAs per SM: the headline shape went from 4.05 to 3.80 us per
    // operation; launches of 64 CTAs already hold four operations at once
    // with two per SM and ran slower with the smaller ring (M256 N512 K2048
    // S4: 3.55 against 3.28 us).
    //
    // Merged chunks: a fused compact plan whose chunks are whole k-blocks
    // gives each CTA two consecutive chunks of its split (all of them where
    // there are two), each in its own accumulator, and the CTA adds the pair
    // before the exchange -- the same sums as one CTA per chunk (the owner
    // adds chunks in pairs), with half the CTAs, each loading twice the K
    // range, and a cluster of half the size.
    // Launched back to back in a graph such CTAs spend less of their time on
    // the fixed parts (set-up, staging, exchange, stores), exchange a
    // quarter of the bytes, and keep three to an SM: on GB300 the headline
    // shape went from 3.61 to 3.21 us per operation in graphs of eight, with
    // the stores made before the wait for the previous grid.
    p.compact = 0;
    p.recv_in_ring = 0;
    // cbn: the compact plan's tile width.  The products of an output element
    // do not depend on it (the same K steps in the same MMA order; checked
    // bitwise on GB300 for widths 64, 128 and 256), so a compact plan may be
    // wider than the plan it stands for and still give the same bits.
    const auto try_compact = [&](int cpc, int cbn) {
        if (N % cbn) return false;
        const int qc = q / cpc;
        const int64_t cctas = row_tiles * (N / cbn) * S * chunks / cpc;
        if (cctas / qc > resident_clusters(qc)) return false;
        const int cols = cbn * cpc;   // tensor-memory columns of a CTA
        const int cshare = share_for(cbn, qc);
        const int cnkb = nkb * cpc;   // k-blocks of a CTA
        // with several chunks a stage holds k-blocks of one chunk: at most
        // the largest power of two dividing a chunk's k-blocks
        const int mk = cpc > 1 ? std::min(kMaxKbs, nkb & -nkb) : kMaxKbs;
        const auto double_buffered = [&](const StageChoice &c) {
            return c.ok && c.stages >= std::min(2, (cnkb + c.kbs - 1) / c.kbs) && (cpc == 1 || nkb % c.kbs == 0);
        };
        StageChoice cc;
        if (qc <= 4 && cols <= 128 && (cctas > resident_clusters(1) / 2 || cpc > 1))
            cc = pick_stages(cbn, cnkb, can3d, qc, cshare, x3, tm, kCompact3SmemLimit, qc > 1, mk);
        if (!double_buffered(cc))
            cc = pick_stages(cbn, cnkb, can3d, qc, cshare, x3, tm, kCompactSmemLimit, qc > 1, mk);
        if (!double_buffered(cc)) return false;
        // the staging area and the receive slots inside the ring, and the
        // shared memory the tensor-memory rule asks for (tmem_fits)
        const size_t in_ring = epi_bytes(cbn) + (qc > 1 ? static_cast<size_t>(qc - 1) * cshare * 16 : 0);
        const size_t tmem_floor = cols <= 128 ? static_cast<size_t>(cols) * 512 : kTmem256Smem;
        const size_t region0 =
            round_up(std::max({cc.stages * stage_bytes(cbn, can3d ? cc.kbs : 1, x3, tm), in_ring, tmem_floor}), 1024);
        if (region0 + 1024 > kCompactSmemLimit || !tmem_fits(cols, region0 + 1024)) return false;
        p.compact = 1;
        p.bn = cbn;
        p.cpc = cpc;
        p.cluster = qc;
        p.share = cshare;
        p.recv_in_ring = qc > 1 ? 1 : 0;
        p.stages = cc.stages;
        p.kbs = can3d ? cc.kbs : 1;
        p.three_d = can3d && p.kbs > 1 ? 1 : 0;
        p.region0 = static_cast<uint32_t>(region0);
        p.smem_bytes = region0 + 1024;
        p.grid = dim3(static_cast<unsigned>(N / cbn), static_cast<unsigned>(row_tiles),
                      static_cast<unsigned>(S * chunks / cpc));
        p.rows_first = 0;
        // two or three CTAs to an SM: as many start beside a running launch as it has CTAs
        p.prefetchers = static_cast<int>(std::min<int64_t>(cctas, 2 * resident_clusters(qc) * qc - cctas));
        if (p.prefetchers < 0) p.prefetchers = 0;
        return true;
    };
    // F32 (3xTF32) plans take the compact layout too (two CTAs per SM: their
    // stages, with the lo halves, are twice as large): on GB300 F32 M96 N512
    // K512 went from 3.98 to 2.36 us per operation in graphs of eight, M256
    // N1024 K2048 S2 from 14.5 to 10.7 us.  They merge pairs of chunks like
    // the 16-bit plans (64-column tiles; the 128-column ones do not fit).
    //
    // A fused plan of 64-column tiles and two chunks first tries 128-column
    // tiles with both chunks in a CTA (two 128-column accumulators, two CTAs
    // per SM): a third less shared-memory traffic per product, half the CTAs.
    // The headline shape went from 3.23 to 2.48 us per operation in graphs of
    // eight calls grouped into one launch.
    //
    // Whole K in a CTA: where the splits are full and their chunks tile them,
    // a fused plan for a launch that follows another may give one CTA every
    // chunk of every split (S x chunks accumulators of 128 columns, at most
    // 512 in all): no cluster and no exchange, the CTA adds its chunks and
    // splits in the owners' order, one CTA per SM with all of its shared
    // memory for the ring.  Only where the compact plan would take more than
    // half the SMs (or there is none): with fewer CTAs a graph of such calls
    // keeps two launches' CTAs on the SMs and ran faster with the compact
    // plan.  A call heading a run launches with its usual plan (alone, its
    // few whole-K CTAs ran up to twice as long: M128 N2048 K4096 S4, 28.6
    // against 14.9 us), and the first call after it converts that launch to
    // whole-K blocks (convert_head).  On GB300, graphs of eight calls went
    // from 5.19 to 4.64 us per call (M128 N2048 K4096 S4), 15.4 to 11.5
    // (M256 N2048 K8192 S4), 9.78 to 6.55 (M512 N1024 K4096 S2) and 11.5 to
    // 8.16 (M128 N4096 K4096 S2); with whole-K blocks M256 N512 K4096 S4 (64
    // compact CTAs) went from 3.09 to 3.60 and the M256 N1024 K2048 S2
    // headline (32) from 2.51 to 2.72, so those keep the compact plan.
    const auto try_whole_k = [&](int cbn) {
        const int units = static_cast<int>(S) * chunks;
        const int cols = cbn * units;
        const int64_t cctas = row_tiles * (N / cbn);
        if (N % cbn || cols > 512 || (cols & (cols - 1)) || cctas > resident_clusters(1)) return false;
        const int cnkb = nkb * units;
        StageChoice cc = pick_stages(cbn, cnkb, can3d, 1, share_for(cbn, 1), x3, tm, kSmemLimit, false,
                                     std::min(kMaxKbs, nkb & -nkb));
        if (!cc.ok || cc.stages < std::min(2, (cnkb + cc.kbs - 1) / cc.kbs) || nkb % cc.kbs != 0) return false;
        p.compact = 1;
        p.bn = cbn;
        p.cpc = units;
        p.cluster = 1;
        p.share = share_for(cbn, 1);
        p.recv_in_ring = 0;
        p.stages = cc.stages;
        p.kbs = can3d ? cc.kbs : 1;
        p.three_d = can3d && p.kbs > 1 ? 1 : 0;
        p.region0 = static_cast<uint32_t>(
            round_up(std::max(cc.stages * stage_bytes(cbn, p.kbs, x3, tm), epi_bytes(cbn)), 1024));
        p.smem_bytes = kSmemLimit;   // alone on its SM: its accumulators may take all 512 columns
        p.grid = dim3(static_cast<unsigned>(N / cbn), static_cast<unsigned>(row_tiles), 1);
        p.rows_first = 0;
        p.prefetchers = 0;
        return true;
    };
    if (compact && tm == kTileM && bn <= 128) {
        const bool mergeable = split_sum == 2 && chunks > 1 && can3d && chunk_len % kb_elems == 0;
        const bool whole = whole_ok && !x3 && split_sum == 2 && S > 1 && can3d && chunk_len % kBlockK == 0 &&
                           K == S * kps && kps == static_cast<int64_t>(chunks) * chunk_len;
        if (!(mergeable && bn == 64 && try_compact(2, 128)) && !(mergeable && bn == 64 && try_compact(2, 64)))
            try_compact(1, bn);
        const int64_t compact_ctas = p.compact ? static_cast<int64_t>(p.grid.x) * p.grid.y * p.grid.z : 0;
        if (whole && (!p.compact || compact_ctas > resident_clusters(1) / 2)) try_whole_k(128);
    }
    return p;
}

}  // namespace

}  // namespace splitk
