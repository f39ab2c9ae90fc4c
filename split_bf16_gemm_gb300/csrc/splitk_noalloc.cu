// splitk_noalloc.cu -- gemm_bt for callers that cannot allocate device memory.
//
// Some hosts hand an operator only its input and output buffers and forbid
// allocation while it runs: plugin interfaces of inference runtimes whose
// execute callback must not call cudaMalloc, or latency-critical loops where
// cudaMalloc's implicit device-wide synchronisation is not acceptable.  Such
// callers cannot provide gemm_bt's workspace, so this file keeps one inside
// the library: a file-scope device array of SPLITK_NOALLOC_MAX_BYTES that
// every GPU loading the library holds until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents (the partials; gemm_bt needs nothing zeroed).  Calls on one stream
// stay ordered (every launch waits for the one before it before its first
// store, inside graph captures too); calls whose executions overlap on the
// GPU (for instance on two streams) race on the array.

#include <cuda_runtime.h>

#include <cstdio>

#include "splitk.h"
#include "splitk_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SPLITK_NOALLOC_MAX_BYTES];

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress with the device current.  It is looked up on every
// call (a lookup; it allocates nothing) rather than kept: after a device
// reset, or once the primary context is torn down and made again, the array
// may sit at another address.  The first call on a device also loads the
// library's device code there.
int scratch_for_current_device(void **ptr)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        splitk::note_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                           "cudaGetSymbolAddress(no-allocation scratch)");
        return SPLITK_ERR_CUDA;
    }
    *ptr = p;
    return SPLITK_OK;
}

}  // namespace

extern "C" int gemm_bt_noalloc(const void *A, const void *B, float *out, int64_t M, int64_t N, int64_t K,
                               int64_t splits, int64_t k_per_split, int dtype, int fused, void *stream)
{
    const int geo = splitk_check_geometry(M, N, K, splits, k_per_split);
    if (geo != SPLITK_OK) return geo;
    const size_t need = gemm_bt_workspace_bytes(M, N, K, splits, k_per_split, fused);
    if (need > static_cast<size_t>(SPLITK_NOALLOC_MAX_BYTES)) {
        char msg[160];
        std::snprintf(msg, sizeof msg, "gemm_bt_noalloc: this shape needs %zu bytes of scratch, the library holds %d",
                      need, SPLITK_NOALLOC_MAX_BYTES);
        splitk::note_message(msg, static_cast<int>(need > 0x7fffffff ? 0x7fffffff : need));
        return SPLITK_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != SPLITK_OK) return st;
    return gemm_bt(A, B, out, scratch, need, M, N, K, splits, k_per_split, dtype, fused, stream);
}
