/*
 * splitk.h -- C ABI of libsplitk: split-K GEMM with prepared, transposed
 * weights, for NVIDIA GB300 (sm_103a).
 *
 * The operation (pages "Aligned shared rows for pipelined NAX on CUDA", section
 * "Contract and correctness", and "Wider consecutive-weight NAX GEMM", section
 * "Launch contract and correctness"):
 *
 *   A        row-major [M,K]          F32, F16 or BF16
 *   B        row-major [N,K]          same element type; the prepared weight,
 *                                     i.e. the transpose of a [K,N] weight
 *   split s  covers k in [s*kps, min((s+1)*kps, K))
 *   partials[s,m,n] = sum_{k in split s} A[m,k] * B[n,k]     F32, [splits,M,N]
 *   out[m,n]        = sum_{s=0}^{splits-1} partials[s,m,n]   F32, [M,N]
 *
 * The second line is the separate accumulation pass the pages run after the
 * partial pass ("an existing accumulation pass produces the final output").
 *
 * Contract enforced by every entry point before any device work:
 *   - M, K and k_per_split are positive multiples of 32; N is a positive
 *     multiple of 64;                                   else SPLITK_ERR_SHAPE
 *   - every split starts below K and the splits cover K, i.e.
 *     splits == ceil(K / k_per_split);                  else SPLITK_ERR_SPLIT
 *   - M, N, K <= SPLITK_MAX_DIM and splits <= SPLITK_MAX_SPLITS
 *     (implementation limits);                           else SPLITK_ERR_SHAPE
 *   - no pointer is NULL;                                else SPLITK_ERR_NULL
 *   - every pointer is 16-byte aligned;                  else SPLITK_ERR_ALIGN
 *   - output byte ranges overlap neither the input ranges nor each other
 *     (A and B may overlap each other: both are only read); else SPLITK_ERR_ALIAS
 *
 * Memory and ownership: every data pointer is a DEVICE pointer on the current
 * CUDA device, owned by the caller, except the host activations and results
 * of gemm_bt_host_batch.  The library allocates no device memory on any call
 * path and keeps no pointer to caller memory for use after a call returns.
 * (Each host thread caches, in host memory, the last tile plans and TMA
 * tensor maps it built; a cached map records an address and a shape and is
 * reused only by a later call with the same address and shape.)
 *
 * Asynchrony and errors: calls enqueue work on `stream` (a cudaStream_t, passed
 * as void*; NULL means the legacy default stream) and return without
 * synchronising.  A non-zero return means nothing was enqueued (validation
 * failed) or the launch itself failed (SPLITK_ERR_CUDA).  No exception and no
 * abort crosses the ABI.  Every wait inside a kernel has a time limit; a wait
 * that runs out sets a device status word, which splitk_get_device_status()
 * reads.  The compute entry points (gemm_splitk_bt, splitk_reduce, gemm_bt,
 * their [K,N] forms, gemm_bt_batch and gemm_bt_noalloc after its first call)
 * may be captured into a CUDA graph.
 *
 * Consecutive launches inside a graph: every launch is a programmatic
 * dependent of the one before it on its stream.  Eagerly, each launch waits
 * for the previous grid to finish before it reads its operands.  While a
 * stream is being captured, the library sees what the next launch depends on
 * (cudaStreamGetCaptureInfo); when that is exactly its own previous launch on
 * the stream, and the new launch reads (A and B; the partials, for the
 * reduce) no byte that any of its launches still able to run writes, the new
 * launch starts loading and multiplying at once and waits for the previous
 * grid only before its first store ("overlap"); if none of them reads or
 * writes what the new launch writes either, it also stores at once and
 * waits only before it finishes, so the grids still finish in launch order.
 * Such a fused launch may also give each thread block two consecutive chunks
 * of its split (all of them where a split has two), each in its own
 * accumulator, added inside the block (the owner adds a split's chunks in
 * pairs too), or, for large shapes with full splits, every chunk of every
 * split.
 * A call that may store early and has the same shape and plan as the launch
 * before it joins that launch instead of adding one: the launch's graph
 * node then computes both calls (up to 8), whose blocks may run in any
 * order; the first such call after a run's first launch may also switch
 * that launch to its own plan (compact, or whole-K).  Its results are
 * bitwise those of the same launch without overlap.
 * Launches that read what an
 * earlier one writes (a chain of GEMMs, the reduce after the partial pass),
 * launches after another kernel or a copy, and launches outside a capture
 * wait as usual.  The decision is made at capture time from the pointers
 * passed; a graph whose nodes are later given other buffers
 * (cudaGraphExecKernelNodeSetParams) must keep the same pattern of overlaps
 * between them, and the calls grouped into one node stay in that node.
 * splitk_set_overlap turns the grouping, or both, off for later captures.
 */
#ifndef SPLITK_H
#define SPLITK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of A and B.  Partials and the output are always F32. */
typedef enum {
    SPLITK_F32 = 0,
    SPLITK_F16 = 1,
    SPLITK_BF16 = 2
} splitk_dtype;

typedef enum {
    SPLITK_OK = 0,
    SPLITK_ERR_NULL = -1,           /* a required pointer is NULL */
    SPLITK_ERR_SHAPE = -2,          /* M,K,kps not positive multiples of 32, N of 64, or too large */
    SPLITK_ERR_SPLIT = -3,          /* splits != ceil(K/kps): a split starts at/after K or K is not covered */
    SPLITK_ERR_ALIAS = -4,          /* an output range overlaps an input or another output */
    SPLITK_ERR_ALIGN = -5,          /* a pointer is not 16-byte aligned */
    SPLITK_ERR_DTYPE = -6,          /* unknown element type */
    SPLITK_ERR_WORKSPACE = -7,      /* workspace smaller than gemm_bt_workspace_bytes() */
    SPLITK_ERR_CUDA = -8,           /* a CUDA runtime call or launch failed */
    SPLITK_ERR_DEVICE_TIMEOUT = -9, /* a kernel's bounded wait ran out (see splitk_get_device_status) */
    SPLITK_ERR_CONFIG = -10         /* an invalid tile override */
} splitk_status;

#define SPLITK_MAX_DIM (1 << 22)
#define SPLITK_MAX_SPLITS 4096
/* Size of the scratch array gemm_bt_noalloc keeps in device memory. */
#define SPLITK_NOALLOC_MAX_BYTES (32 << 20)

/* Checks the contract's shape and split rules only (no pointers, no device
 * work).  Returns SPLITK_OK, SPLITK_ERR_SHAPE or SPLITK_ERR_SPLIT; the shape
 * rule is checked first. */
int splitk_check_geometry(int64_t M, int64_t N, int64_t K, int64_t splits,
                          int64_t k_per_split);

/* The partial pass: partials[s,m,n] = sum over split s of A[m,k]*B[n,k].
 *   A         device, [M,K] row-major, element type `dtype`
 *   B         device, [N,K] row-major, element type `dtype`
 *   partials  device, [splits,M,N] row-major F32; fully overwritten
 * BF16/F16 operands run on the tensor cores (tcgen05, F32 accumulate in tensor
 * memory, native operands).  F32 operands run on the tensor cores too, each
 * product as three TF32 products: x = hi + lo, where hi is the F32 operand as
 * loaded, which the tensor cores read as TF32 by dropping its 13 low fraction
 * bits (its top 19 bits; measured on GB300: truncation, not rounding), and
 * lo = x - (x with those 13 bits cleared), exact in F32; hi*lo + lo*hi +
 * hi*hi, relative error per product about 2^-21.  Each element is a sum in
 * F32 whose order is fixed for a given shape. */
int gemm_splitk_bt(const void *A, const void *B, float *partials, int64_t M,
                   int64_t N, int64_t K, int64_t splits, int64_t k_per_split,
                   int dtype, void *stream);

/* Weight preparation (pages: "Wider consecutive-weight NAX GEMM", section
 * "Performance method" -- the transposed layout is prepared once, outside
 * timing, and kept resident): B[n,k] = W[k,n].
 *   W  device, [K,N] row-major, element type `dtype` (bits copied as they are)
 *   B  device, [N,K] row-major, same type; fully overwritten
 * K a positive multiple of 32 and N of 64 (the GEMM's contract for B),
 * 16-byte aligned pointers, no overlap; else SPLITK_ERR_SHAPE / _DTYPE /
 * _NULL / _ALIGN / _ALIAS before any device work. */
int splitk_prepare_bt(const void *W, void *B, int64_t K, int64_t N, int dtype,
                      void *stream);

/* The accumulation pass: out[i] = (((P[0][i] + P[1][i]) + P[2][i]) + ...) in
 * F32, in split order s = 0..splits-1.
 *   partials  device, [splits,M,N] F32, read only
 *   out       device, [M,N] F32; fully overwritten
 * Requires M, N >= 1, splits >= 1, 16-byte aligned pointers and no overlap
 * between the two ranges. */
int splitk_reduce(const float *partials, float *out, int64_t splits, int64_t M,
                  int64_t N, void *stream);

/* Bytes of device workspace gemm_bt needs: the F32 partials [splits,M,N],
 * splits*M*N*4 bytes.  The same size serves every value of `fused`.  Returns
 * 0 for a geometry that breaks the contract. */
size_t gemm_bt_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t splits,
                               int64_t k_per_split, int fused);

/* Zeroes a workspace (cudaMemsetAsync on `stream`).  gemm_bt needs no
 * particular workspace contents (every byte it reads it wrote in the same
 * call); this gives callers a defined starting state. */
int gemm_bt_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* One call: the partial pass then the accumulation pass, on one stream.
 *   out        device, [M,N] F32; fully overwritten
 *   workspace  device, >= gemm_bt_workspace_bytes() bytes, caller-owned
 *              scratch; may not overlap A, B or out.
 *   fused      0: two kernels (gemm_splitk_bt, then splitk_reduce); the
 *                 workspace then holds the partials [splits,M,N] in its
 *                 first bytes;
 *              1: one kernel where the tile plan holds all of a tile's
 *                 splits in one resident thread-block cluster: the splits
 *                 are summed inside the launch, over distributed shared
 *                 memory, and the partials are not kept.  Where it cannot
 *                 (too many splits for one cluster, or more tiles than
 *                 resident clusters), the call runs the two kernels of 0,
 *                 which measured faster there than summing through global
 *                 memory.  splitk_describe_launch reports which;
 *              3: as 1, and the workspace also holds the partials afterwards.
 * For a given shape, `out` (and the partials, where kept) are bitwise the
 * same for every value of `fused`. */
int gemm_bt(const void *A, const void *B, float *out, void *workspace,
            size_t workspace_bytes, int64_t M, int64_t N, int64_t K,
            int64_t splits, int64_t k_per_split, int dtype, int fused,
            void *stream);

/* The same two operations with the weight in its own [K,N] layout, the other
 * layout the pages keep resident ("Wider consecutive-weight NAX GEMM",
 * section "Performance method": both layouts uploaded once); no preparation
 * step.
 *   W  device, [K,N] row-major, element type `dtype`; B[n,k] = W[k,n]
 * Every other argument, the contract and the checks are those of
 * gemm_splitk_bt and gemm_bt with B = W^T, and for BF16/F16 the results too
 * (bitwise): the tensor cores read W N-contiguous (MN-major operand).  F32
 * operands with W run exact F32 FMA on the CUDA cores (no fused variant: the
 * two-kernel path runs for every `fused`). */
int gemm_splitk_kn(const void *A, const void *W, float *partials, int64_t M,
                   int64_t N, int64_t K, int64_t splits, int64_t k_per_split,
                   int dtype, void *stream);
int gemm_kn(const void *A, const void *W, float *out, void *workspace,
            size_t workspace_bytes, int64_t M, int64_t N, int64_t K,
            int64_t splits, int64_t k_per_split, int dtype, int fused,
            void *stream);

/* gemm_bt for callers that cannot allocate device memory.  The paper has no
 * counterpart of this entry point; it exists for hosts that hand an operator
 * only its input and output buffers and forbid allocation while it runs (the
 * execute callback of an inference-runtime plugin, for one) and for loops
 * where cudaMalloc's implicit device synchronisation is not acceptable.
 *   A, B, out, M, N, K, splits, k_per_split, dtype, fused, stream
 *              as for gemm_bt; no workspace argument.
 * Instead of a caller workspace it uses a scratch array of
 * SPLITK_NOALLOC_MAX_BYTES (32 MiB) that the library keeps in device memory;
 * every GPU that loads the library holds that array until the process exits.
 * A shape whose gemm_bt_workspace_bytes() exceeds it is rejected with
 * SPLITK_ERR_WORKSPACE before any device work (splitk_last_error() gives the
 * sizes).  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.  Each call looks up the array's device
 * address on the current device (cudaGetSymbolAddress, a lookup that
 * allocates nothing); the first call on a device also loads the library's
 * device code there, so make that first call before any stream capture.
 * Every call on a device shares the one array and leaves its contents behind
 * (the partials).  Calls whose executions overlap on the GPU (on different
 * streams, say) race on the array and must not be issued. */
int gemm_bt_noalloc(const void *A, const void *B, float *out, int64_t M,
                    int64_t N, int64_t K, int64_t splits, int64_t k_per_split,
                    int dtype, int fused, void *stream);

/* `count` independent operations out_i = gemm_bt(A_i, B_i) of one shape on
 * device buffers, enqueued on `stream` in as few launches as the plan
 * allows.  The pages time eight complete operations per replay ("pack 8":
 * "Aligned shared rows for pipelined NAX on CUDA", section "Measurement
 * protocol"); outside a graph capture this call gives such a pack the
 * grouped launches a capture would.
 *   A, B, out   host arrays of `count` DEVICE pointers: activations [M,K],
 *               prepared weights [N,K] (entries may repeat, as may A's) and
 *               outputs [M,N] F32, each fully overwritten
 *   workspace   device, >= gemm_bt_workspace_bytes() bytes: scratch for the
 *               operations that run the two kernels, used one after another
 *   count       1 .. 65536
 *   fused       0 or 1 (as for gemm_bt; fused = 1 calls whose splits are
 *               summed inside the launch run up to 8 to a launch, BF16/F16
 *               with a compact plan; everything else one gemm_bt each)
 * Every result is bitwise that of gemm_bt(fused) on the same operands.
 * Returns as gemm_bt's validation would for each operation, plus
 * SPLITK_ERR_CONFIG for count outside [1, 65536] or fused not 0 or 1, and
 * SPLITK_ERR_ALIAS when an output overlaps another output, an input or the
 * workspace; nothing is enqueued unless every operation passes. */
int gemm_bt_batch(const void *const *A, const void *const *B, float *const *out,
                  int64_t count, void *workspace, size_t workspace_bytes,
                  int64_t M, int64_t N, int64_t K, int64_t splits,
                  int64_t k_per_split, int dtype, int fused, void *stream);

/* Device staging bytes gemm_bt_host_batch needs for `count` operations of
 * this shape: count A slots [M,K], count output slots [M,N] F32 and one
 * gemm_bt workspace.  Returns 0 for a rejected geometry or element type, or
 * count outside [1, 65536]. */
size_t gemm_bt_host_staging_bytes(int64_t count, int64_t M, int64_t N,
                                  int64_t K, int64_t splits,
                                  int64_t k_per_split, int dtype);

/* `count` operations out_i = gemm_bt(A_i, B_i) whose activations and results
 * live in HOST memory.  The pages time operands already on the device; this
 * entry point adds the copies a serving loop needs, pipelined so that they
 * overlap the kernels.
 *   A_host     host, [count,M,K] elements of `dtype`, operation i at
 *              i*M*K; read by the copy engine (page-locked memory lets the
 *              copies run asynchronously; any memory cudaMemcpyDefault
 *              accepts works)
 *   B          host array of `count` DEVICE pointers, each a prepared weight
 *              [N,K] (16-byte aligned; entries may repeat)
 *   out_host   host, [count,M,N] F32; fully overwritten once `stream`
 *              reaches the end of the call's work
 *   staging    device, >= gemm_bt_host_staging_bytes(), 16-byte aligned,
 *              overlapping no B
 *   fused      as for gemm_bt (0, 1 or 3)
 *   ops_per_copy  operations moved by one copy each way; 0 lets the library
 *              choose (at least 4 MiB of A per copy, at most half the batch)
 * Every operation is bitwise the gemm_bt result for its operands.  With
 * fused = 1, 16-bit operands and a shape whose splits are summed inside the
 * launch, the operations of a group run as one launch (up to 8 of them; the
 * same tiles and sums as one call each); otherwise one gemm_bt each.  The copy
 * in of group g+1 and the copy out of group g-1 run on two library streams
 * while group g computes on `stream`, and `stream` waits for the last copy
 * out, so synchronising `stream` completes the batch.  Host buffers must stay
 * valid until then.  The copy in waits for the end of the previous call on
 * the same staging (the library keeps one event per staging buffer, for the
 * 32 most recently used), or, for a staging it has not seen, for the work
 * already on `stream`: calls that alternate two staging buffers overlap one
 * batch's copy in with the previous batch's kernels.  On one stream a call's
 * kernels still follow the previous call's copy out (stream order); calls
 * that alternate two streams as well also overlap that copy out with the
 * next batch's kernels.  Between calls the
 * staging belongs to them: other work must not write it, and one staging is
 * used with one stream (its workspace part is used in stream order).
 * The first call on a device creates those two streams and four events (kept
 * until exit); a process-wide mutex serialises the enqueueing of concurrent
 * calls.  Returns as gemm_bt's validation would (plus SPLITK_ERR_CONFIG for
 * count outside [1, 65536] or ops_per_copy < 0, SPLITK_ERR_WORKSPACE for a
 * small staging, SPLITK_ERR_ALIAS when A_host and out_host overlap or the
 * staging overlaps a B or a host range) before enqueueing anything. */
int gemm_bt_host_batch(const void *A_host, const void *const *B,
                       float *out_host, int64_t count, void *staging,
                       size_t staging_bytes, int64_t M, int64_t N, int64_t K,
                       int64_t splits, int64_t k_per_split, int dtype,
                       int fused, int64_t ops_per_copy, void *stream);

/* Split count for a shape.  The pages sweep 1, 2, 4, 8 and 16 splits of fixed
 * shapes ("Aligned shared rows for pipelined NAX on CUDA", section
 * "Measurement protocol"; "Wider consecutive-weight NAX GEMM", section
 * "Performance method"); these two entry points pick among the same
 * candidates.  For a candidate n, k_per_split = ceil(K/n) rounded up to a
 * multiple of 32 and splits = ceil(K/k_per_split) (below n when K is short).
 *
 * splitk_choose_splits: the library's cost model of gemm_bt with `fused`
 * (the tile planner's estimate plus the reduce for the two-kernel path); no
 * device work.  Writes the cheapest legal (splits, k_per_split) and, when
 * model_us is not NULL, model_us[0..4] = the estimate in microseconds per
 * call for candidates 1, 2, 4, 8, 16 (-1 for an illegal one).  M and K positive
 * multiples of 32, N of 64 (else SPLITK_ERR_SHAPE), a known dtype
 * (SPLITK_ERR_DTYPE), fused in {0, 1, 3} (SPLITK_ERR_CONFIG), non-NULL
 * outputs (SPLITK_ERR_NULL). */
int splitk_choose_splits(int64_t M, int64_t N, int64_t K, int dtype, int fused,
                         int64_t *splits, int64_t *k_per_split,
                         double *model_us);

/* splitk_autotune_splits: measures each candidate on the caller's buffers
 * (A, B, out, workspace as for gemm_bt) and writes the fastest legal
 * (splits, k_per_split).  Per candidate: one untimed call, then a CUDA graph
 * of `reps` calls (1..1000) replayed three times between CUDA events on a
 * private stream that first waits for the work already on `stream`.
 * us[0..4], when not NULL, receive the microseconds per call of candidates
 * 1, 2, 4, 8, 16 (-1 where a candidate was not run: its workspace does not
 * fit `workspace_bytes`, or it repeats an earlier candidate's split count).
 * Every candidate's arguments are checked before anything is enqueued (the
 * statuses of gemm_bt; SPLITK_ERR_WORKSPACE if no candidate fits).  On
 * return the private stream has finished, `out` holds the chosen split's
 * result and `stream` is ordered after it.  The inputs are
 * read repeatedly, so they sit in L2 when they fit there: the timings rank
 * the candidates, they are not cold-cache figures.  Not capturable. */
int splitk_autotune_splits(const void *A, const void *B, float *out,
                           void *workspace, size_t workspace_bytes, int64_t M,
                           int64_t N, int64_t K, int dtype, int fused,
                           int reps, void *stream, int64_t *splits,
                           int64_t *k_per_split, float *us);

/* Reads and clears the device status word on the current device,
 * synchronising `stream` first.  Returns SPLITK_OK, SPLITK_ERR_DEVICE_TIMEOUT
 * (since the last call a kernel's bounded wait ran out, or a launch met a tile
 * configuration it cannot run; that launch's outputs are not valid) or
 * SPLITK_ERR_CUDA. */
int splitk_get_device_status(void *stream);

/* What the most recent SPLITK_ERR_CUDA on the calling host thread came from:
 * the failing call and CUDA's name and description of its error.  The string
 * is owned by the library and stays valid until the thread's next failure. */
const char *splitk_last_error(void);

/* A short, static description of a status code. */
const char *splitk_status_string(int status);

/* Tile-shape override for tuning: every later tensor-core launch uses tile
 * width `bn` (64, 128 or 256; must divide N, else the automatic choice is
 * kept), `chunks` thread blocks per split along K (1, 2, 4 or 8; fewer when
 * the shared memory of that many does not fit) and `kblocks_per_stage`
 * 64-wide k-blocks per pipeline stage (1, 2 or 4; more than 1 only when K and
 * k_per_split are multiples of 64).  Zero keeps the automatic choice for that
 * item.  Process-wide; not thread-safe against concurrent launches.  Returns
 * SPLITK_OK or SPLITK_ERR_CONFIG. */
int splitk_set_tile_override(int bn, int chunks, int kblocks_per_stage);

/* Describes the launch gemm_bt would make, without launching: info[0..25] =
 * {path (0 tensor-core, 2 tensor-core 3xTF32 for F32), bn, chunks, chunk_len, stages,
 *  cluster_size (chunks, or splits * chunks), grid_x, grid_y, grid_z,
 *  dynamic_smem_bytes,
 *  fused_in_kernel (0/1), kernels_per_call, kblocks_per_stage,
 *  three_d_loads (0/1), split_sum (0 none, 2 inside the thread-block
 *  cluster; a fused call whose splits do not fit one resident cluster
 *  reports the two-kernel launch, fused_in_kernel 0), prefetchers (fused calls
 *  only: CTAs that fit beside a running launch and prefetch A and B into L2
 *  before the dependency wait), rows_first (1: grid x walks the 128-row tiles
 *  and grid y the column tiles, so grid_x and grid_y are swapped; chosen for
 *  launches of more than one wave with M < N whose B slab per split,
 *  N * k_per_split elements, is over 32 MB), tile_m (rows of A per thread
 *  block: 128, or 256 for BN 256 plans with one block per tile, no cluster
 *  chosen when it saves waves; grid_x or grid_y
 *  then counts 256-row tiles),
 *  compact (1: the call's tensor-core launch, captured into a graph, when it
 *  starts beside the launch before it or heads such a run, takes the compact
 *  layout: the same tiles, chunks and sums, a stage ring cut so that two or
 *  three thread blocks fit on an SM, the peers' shares received inside the
 *  ring; one-wave plans),
 *  compact_stages, compact_kblocks_per_stage, compact_dynamic_smem_bytes,
 *  compact_chunks_per_block (1, or two consecutive chunks of a split in one
 *  thread block, each in its own accumulator, added before the exchange:
 *  the same sums, since a split's chunks are added in pairs; or, more than
 *  chunks, every chunk of every split in one block of 128 x 128, no cluster and one block per SM, which
 *  adds each split's chunks and then the splits in the same order: fused
 *  16-bit calls whose splits are full and whose chunks tile them, where the
 *  compact plan would take more than half the SMs), compact_cluster_size,
 *  compact_grid_z,
 *  compact_bn (the compact plan's tile width, which may be wider than bn:
 *  the products of an output element do not depend on it)
 *  (0 when compact is 0).  The compact fields describe a call that starts
 *  beside the launch before it; the first call of a run launches without
 *  whole-K blocks, and the next call that takes them converts that launch
 *  and joins it}; `info` must hold 26 ints.
 * Returns a status as gemm_bt's validation would (pointers are not checked). */
int splitk_describe_launch(int64_t M, int64_t N, int64_t K, int64_t splits,
                           int64_t k_per_split, int dtype, int fused,
                           int *info);

/* Self-test of the bounded-wait machinery: launches one block that waits on a
 * barrier nothing ever completes, with a limit of `limit_ns` nanoseconds
 * (clamped to [1e3, 1e9]), synchronises `stream`, and returns what
 * splitk_get_device_status() then reads (SPLITK_ERR_DEVICE_TIMEOUT expected). */
int splitk_selftest_bounded_wait(int64_t limit_ns, void *stream);

/* Self-test of the tensor-core kernel's own time-out path: one fused launch
 * (arguments as for gemm_bt with fused = 1, no workspace; the shape must sum
 * its splits inside the launch, else SPLITK_ERR_CONFIG) whose wait for the
 * final accumulator gives up at once: the warps that wait for it test it
 * once, before the MMA issuer has finished, as a wait that ran out would.  The
 * kernel then records the time-out, still sends and awaits every cluster
 * message, waits for the MMAs (normal limit) before it frees its tensor
 * memory, and finishes; `out` is not valid.  Synchronises `stream` and
 * returns what splitk_get_device_status() reads (SPLITK_ERR_DEVICE_TIMEOUT
 * expected).  At that wait every TMA load of the launch has landed, and the
 * waits after it keep their normal limits, so no copy is in flight when a
 * block exits. */
int splitk_selftest_kernel_timeout(const void *A, const void *B, float *out,
                                   int64_t M, int64_t N, int64_t K,
                                   int64_t splits, int64_t k_per_split,
                                   int dtype, void *stream);

/* What the library does with consecutive independent calls inside a graph
 * capture (see the top of this header), for every later call of the
 * process: 2 (the default) overlap them and group them into one launch
 * where they can be; 1 overlap them only (one launch per call); 0 neither
 * (every launch waits for the one before).  Launches already captured keep
 * what was decided for them.  Returns SPLITK_OK or SPLITK_ERR_CONFIG. */
int splitk_set_overlap(int mode);

/* What the calling host thread's most recent tensor-core launch did:
 * info[0..10] = {overlap (0: it waited for the previous grid before loading;
 * 1: it loaded before that grid finished and waited before its first store;
 * 2: it also stored before, waiting only before it finished), compact (its
 * ring was cut so that two or three of its thread blocks fit on an SM,
 * taken for such launches and for the first of a capture, when a one-wave
 * plan allows it), capturing (the stream was being captured), bn, chunks,
 * stages, kblocks_per_stage, dynamic_smem_bytes, chunks_per_block (1, or
 * two consecutive chunks of a split, each in its own accumulator and added
 * inside the block: the same sums; more than chunks: every chunk of every
 * split, no cluster), cluster_size, group (the calls
 * the launch computes so far: 1, or more where the call joined the launch
 * of the calls before it)}.  `info` must hold 11 ints.  Diagnostic;
 * returns SPLITK_OK or SPLITK_ERR_NULL. */
int splitk_last_launch(int *info);

#ifdef __cplusplus
}
#endif

#endif /* SPLITK_H */
