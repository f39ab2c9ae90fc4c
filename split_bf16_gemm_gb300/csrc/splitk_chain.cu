// splitk_chain.cu -- which tensor-core launches may start before the launch
// before them has finished.
//
// Every launch of this library is a programmatic dependent of the one before
// it on its stream.  Normally a launch waits (griddepcontrol.wait) for that
// grid to finish before it reads its operands, because the grid may have
// written them.  Inside a CUDA graph capture the library can see what a new
// launch depends on (cudaStreamGetCaptureInfo): when that is exactly the node
// of its own previous launch, it knows which device memory every launch of
// the chain since then writes.  If the new launch reads none of it, it may
// load and multiply before the previous grid ends, waiting only before its
// first store ("overlap").  If no launch of the chain reads or writes what
// the new one writes either, it stores at once too and waits for the
// previous grid only before it finishes ("store early"): the grids still
// finish in launch order.
//
// Which launches can still be running when an overlapping launch starts:
// a "head" -- a launch that waits at its start and lets the next grid start
// only after that wait returned -- guarantees that everything before it has
// finished when its successor starts; every other launch (an overlapping
// one, or a reduce after a partial pass, which waits for its partials but
// lets the next grid start at once) lets the next grid start as soon as its
// own CTAs have started.  So a launch can meet
// every launch from the last head on, and the window it is checked against
// is exactly that run: [head, ..., previous].  Every launch also waits for
// the previous grid before it finishes, so the grids finish in order, and
// before its first store unless nothing in that run reads or writes what it
// writes, so no launch overwrites what an earlier one still reads or writes.
//
// Eager launches (no capture) always wait: the library cannot see what else
// the caller put on the stream.  splitk_set_overlap(0) turns the mechanism off.

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "splitk_internal.h"

namespace splitk {
namespace {

constexpr int kChains = 16;    // capture sequences followed at once (least recently used replaced)
constexpr int kWindow = 32;    // launches a new one is checked against, at most

// a launch's byte ranges: two of each kind per call, for every call grouped into it
constexpr int kEntrySpans = kMaxSpans * kMaxGroup;

struct Entry {
    cudaGraphNode_t node;
    Span reads[kEntrySpans], writes[kEntrySpans];
    int n_reads, n_writes;
};

struct Chain {
    unsigned long long id = 0;
    bool used = false;
    uint64_t stamp = 0;
    int n = 0;                 // entries e[0..n-1]; e[0] is the head
    Entry e[kWindow];
};

std::mutex g_mu;
Chain g_chains[kChains];
uint64_t g_clock = 0;
std::atomic<int> g_mode{2};

Chain *find_chain(unsigned long long id)
{
    for (Chain &c : g_chains)
        if (c.used && c.id == id) return &c;
    return nullptr;
}

Chain *make_chain(unsigned long long id)
{
    Chain *victim = &g_chains[0];
    for (Chain &c : g_chains) {
        if (!c.used) {
            victim = &c;
            break;
        }
        if (c.stamp < victim->stamp) victim = &c;
    }
    victim->used = true;
    victim->id = id;
    victim->n = 0;
    return victim;
}

bool meets(const Span &a, const Span &b) { return a.lo < b.hi && b.lo < a.hi; }

}  // namespace

void set_overlap_mode(int mode) { g_mode.store(mode); }
bool overlap_enabled() { return g_mode.load() >= 1; }
bool grouping_enabled() { return g_mode.load() >= 2; }

namespace {
thread_local LaunchRecord t_last = {};
}
void note_launch(const LaunchRecord &r) { t_last = r; }
LaunchRecord last_launch() { return t_last; }

ChainGuard::ChainGuard(cudaStream_t stream, const Span *reads, int n_reads, const Span *writes, int n_writes)
    : stream_(stream)
{
    if (n_reads > kMaxSpans || n_writes > kMaxSpans) return;   // not followed: the launch waits
    n_reads_ = n_reads;
    n_writes_ = n_writes;
    for (int r = 0; r < n_reads; ++r) reads_[r] = reads[r];
    for (int w = 0; w < n_writes; ++w) writes_[w] = writes[w];
    if (!overlap_enabled()) return;
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    unsigned long long id = 0;
    const cudaGraphNode_t *deps = nullptr;
    size_t nd = 0;
    if (cudaStreamGetCaptureInfo(stream, &st, &id, nullptr, &deps, nullptr, &nd) != cudaSuccess ||
        st != cudaStreamCaptureStatusActive)
        return;
    lock_ = std::unique_lock<std::mutex>(g_mu);
    capturing_ = true;
    id_ = id;
    fresh_ = true;
    Chain *c = find_chain(id);
    if (!c || c->n == 0 || nd != 1 || deps[0] != c->e[c->n - 1].node) return;   // not after our own launch
    fresh_ = false;
    dep_ = deps[0];
    for (int i = 0; i < c->n; ++i)
        for (int w = 0; w < c->e[i].n_writes; ++w)
            for (int r = 0; r < n_reads; ++r)
                if (meets(c->e[i].writes[w], reads[r])) return;   // reads what a running launch may write
    if (c->n >= kWindow) {
        fresh_ = true;   // a long run: this launch waits and starts a new window
        return;
    }
    overlap_ = true;
    store_early_ = true;
    for (int i = 0; i < c->n && store_early_; ++i)
        for (int w = 0; w < n_writes && store_early_; ++w) {
            for (int x = 0; x < c->e[i].n_writes; ++x)
                if (meets(c->e[i].writes[x], writes[w])) store_early_ = false;
            for (int x = 0; x < c->e[i].n_reads; ++x)
                if (meets(c->e[i].reads[x], writes[w])) store_early_ = false;
        }
}

void ChainGuard::commit(bool launched, bool head)
{
    if (!capturing_) return;
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    unsigned long long id = 0;
    const cudaGraphNode_t *deps = nullptr;
    size_t nd = 0;
    Chain *c = find_chain(id_);
    const bool ok = launched &&
                    cudaStreamGetCaptureInfo(stream_, &st, &id, nullptr, &deps, nullptr, &nd) == cudaSuccess &&
                    st == cudaStreamCaptureStatusActive && id == id_ && nd == 1;
    if (!ok) {
        if (c) c->used = false;   // unknown state: the next launch waits and starts afresh
        return;
    }
    if (head) {
        if (!c) c = make_chain(id_);
        c->n = 0;                  // everything before it has finished when its successor starts
    } else if (!c || fresh_ || c->n >= kWindow) {
        // A launch that lets its successor start early can only extend a run
        // that a head began: after anything else (another kernel, a copy) its
        // successor could meet work the library cannot see.  The next launch
        // then waits and heads a new run.
        if (c) c->used = false;
        return;
    }
    Entry &e = c->e[c->n++];
    e.node = deps[0];
    e.n_reads = n_reads_;
    e.n_writes = n_writes_;
    for (int r = 0; r < n_reads_; ++r) e.reads[r] = reads_[r];
    for (int w = 0; w < n_writes_; ++w) e.writes[w] = writes_[w];
    c->stamp = ++g_clock;
}

void ChainGuard::commit_joined()
{
    if (!capturing_) return;
    Chain *c = find_chain(id_);
    if (!c || c->n == 0) return;
    Entry &e = c->e[c->n - 1];
    if (e.n_reads + n_reads_ > kEntrySpans || e.n_writes + n_writes_ > kEntrySpans) {
        c->used = false;   // cannot record it: the next launch waits and starts afresh
        return;
    }
    for (int r = 0; r < n_reads_; ++r) e.reads[e.n_reads++] = reads_[r];
    for (int w = 0; w < n_writes_; ++w) e.writes[e.n_writes++] = writes_[w];
    c->stamp = ++g_clock;
}

}  // namespace splitk
