"""ctypes binding of libsplitk's C ABI (include/splitk.h), with the same names.

Argument marshalling only: tensors become device pointers (``data_ptr()``),
streams become ``cudaStream_t`` handles, a non-zero status becomes a
``SplitKError``.  Every step of the computation runs in libsplitk's kernels;
there is no fallback of any kind, and every call fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsplitk.so")

# Element types and status codes, as in include/splitk.h.
F32, F16, BF16 = 0, 1, 2
OK = 0
ERR_NULL, ERR_SHAPE, ERR_SPLIT, ERR_ALIAS, ERR_ALIGN = -1, -2, -3, -4, -5
ERR_DTYPE, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_CONFIG = -6, -7, -8, -9, -10

EXPORTS = (
    "splitk_check_geometry", "gemm_splitk_bt", "splitk_reduce", "gemm_bt_workspace_bytes",
    "gemm_bt", "splitk_get_device_status", "splitk_status_string", "splitk_set_tile_override",
    "splitk_describe_launch", "splitk_selftest_bounded_wait", "splitk_last_error",
    "gemm_bt_workspace_init", "gemm_bt_noalloc", "splitk_prepare_bt",
    "gemm_bt_host_staging_bytes", "gemm_bt_host_batch", "splitk_choose_splits", "splitk_autotune_splits",
    "gemm_splitk_kn", "gemm_kn", "splitk_set_overlap", "splitk_last_launch", "splitk_selftest_kernel_timeout",
    "gemm_bt_batch",
)
NOALLOC_MAX_BYTES = 32 << 20   # SPLITK_NOALLOC_MAX_BYTES

_lock = threading.Lock()
_lib = None


class SplitKError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: status {status} ({status_string(status)})"
        if status == ERR_CUDA:
            msg += ": " + last_error()
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """The loaded libsplitk (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libsplitk is not built ({LIB_PATH} missing); "
                                   "run split_bf16_gemm_gb300.build()")
            L = ctypes.CDLL(LIB_PATH)
            i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
            L.splitk_check_geometry.argtypes = [i64] * 5
            L.gemm_splitk_bt.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
            L.splitk_reduce.argtypes = [vp, vp, i64, i64, i64, vp]
            L.gemm_bt_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i32]
            L.gemm_bt_workspace_bytes.restype = sz
            L.gemm_bt.argtypes = [vp, vp, vp, vp, sz, i64, i64, i64, i64, i64, i32, i32, vp]
            L.gemm_bt_batch.argtypes = [vp, vp, vp, i64, vp, sz, i64, i64, i64, i64, i64, i32, i32, vp]
            L.gemm_splitk_kn.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
            L.gemm_kn.argtypes = [vp, vp, vp, vp, sz, i64, i64, i64, i64, i64, i32, i32, vp]
            L.splitk_get_device_status.argtypes = [vp]
            L.splitk_status_string.argtypes = [i32]
            L.splitk_status_string.restype = ctypes.c_char_p
            L.splitk_set_tile_override.argtypes = [i32, i32, i32]
            L.splitk_describe_launch.argtypes = [i64, i64, i64, i64, i64, i32, i32, vp]
            L.splitk_selftest_bounded_wait.argtypes = [i64, vp]
            L.gemm_bt_workspace_init.argtypes = [vp, sz, vp]
            L.gemm_bt_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, i32, vp]
            L.splitk_prepare_bt.argtypes = [vp, vp, i64, i64, i32, vp]
            L.gemm_bt_host_staging_bytes.argtypes = [i64] * 6 + [i32]
            L.gemm_bt_host_staging_bytes.restype = sz
            L.gemm_bt_host_batch.argtypes = [vp, vp, vp, i64, vp, sz, i64, i64, i64, i64, i64, i32, i32,
                                             i64, vp]
            L.splitk_choose_splits.argtypes = [i64, i64, i64, i32, i32, vp, vp, vp]
            L.splitk_autotune_splits.argtypes = [vp, vp, vp, vp, sz, i64, i64, i64, i32, i32, i32, vp, vp, vp, vp]
            L.splitk_last_error.argtypes = []
            L.splitk_set_overlap.argtypes = [i32]
            L.splitk_last_launch.argtypes = [vp]
            L.splitk_selftest_kernel_timeout.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
            L.splitk_last_error.restype = ctypes.c_char_p
            for name in ("splitk_check_geometry", "gemm_splitk_bt", "splitk_reduce", "gemm_bt",
                         "gemm_splitk_kn", "gemm_kn",
                         "gemm_bt_workspace_init", "gemm_bt_noalloc", "splitk_prepare_bt",
                         "gemm_bt_host_batch", "splitk_choose_splits", "splitk_autotune_splits",
                         "splitk_get_device_status", "splitk_set_tile_override",
                         "splitk_describe_launch", "splitk_selftest_bounded_wait", "splitk_set_overlap",
                         "splitk_last_launch", "splitk_selftest_kernel_timeout"):
                getattr(L, name).restype = i32
            _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(dtype) -> int:
    """Element-type code from a name ('bf16', 'f16', 'f32'), a torch dtype or an int."""
    if isinstance(dtype, int):
        return dtype
    if isinstance(dtype, str):
        return {"f32": F32, "f16": F16, "bf16": BF16}[dtype]
    import torch

    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[dtype]


def _check(status: int, where: str) -> None:
    if status != OK:
        raise SplitKError(status, where)


def status_string(status: int) -> str:
    return lib().splitk_status_string(status).decode()


splitk_status_string = status_string


def last_error() -> str:
    """The failing CUDA call behind the calling thread's latest ERR_CUDA."""
    return lib().splitk_last_error().decode()


splitk_last_error = last_error


def splitk_check_geometry(M, N, K, splits, k_per_split) -> int:
    """Contract status of a geometry (0 legal, ERR_SHAPE or ERR_SPLIT); never raises."""
    return lib().splitk_check_geometry(M, N, K, splits, k_per_split)


def gemm_splitk_bt(A, B, partials, M, N, K, splits, k_per_split, dtype, stream=None) -> None:
    _check(lib().gemm_splitk_bt(_ptr(A), _ptr(B), _ptr(partials), M, N, K, splits, k_per_split,
                                dtype_code(dtype), _stream(stream)), "gemm_splitk_bt")


def gemm_splitk_kn(A, W, partials, M, N, K, splits, k_per_split, dtype, stream=None) -> None:
    """gemm_splitk_bt with the weight W in its [K,N] layout."""
    _check(lib().gemm_splitk_kn(_ptr(A), _ptr(W), _ptr(partials), M, N, K, splits, k_per_split,
                                dtype_code(dtype), _stream(stream)), "gemm_splitk_kn")


def gemm_kn(A, W, out, workspace, workspace_bytes, M, N, K, splits, k_per_split, dtype, fused=0,
            stream=None) -> None:
    """gemm_bt with the weight W in its [K,N] layout."""
    _check(lib().gemm_kn(_ptr(A), _ptr(W), _ptr(out), _ptr(workspace), workspace_bytes, M, N, K,
                         splits, k_per_split, dtype_code(dtype), fused, _stream(stream)), "gemm_kn")


def splitk_prepare_bt(W, B, K, N, dtype, stream=None) -> None:
    """Weight preparation: B[n,k] = W[k,n] (W row-major [K,N], B row-major [N,K])."""
    _check(lib().splitk_prepare_bt(_ptr(W), _ptr(B), K, N, dtype_code(dtype), _stream(stream)),
           "splitk_prepare_bt")


def splitk_reduce(partials, out, splits, M, N, stream=None) -> None:
    _check(lib().splitk_reduce(_ptr(partials), _ptr(out), splits, M, N, _stream(stream)),
           "splitk_reduce")


def gemm_bt_workspace_bytes(M, N, K, splits, k_per_split, fused=0) -> int:
    return int(lib().gemm_bt_workspace_bytes(M, N, K, splits, k_per_split, fused))


def gemm_bt_workspace_init(workspace, workspace_bytes, stream=None) -> None:
    _check(lib().gemm_bt_workspace_init(_ptr(workspace), workspace_bytes, _stream(stream)),
           "gemm_bt_workspace_init")


def gemm_bt(A, B, out, workspace, workspace_bytes, M, N, K, splits, k_per_split, dtype, fused=0,
            stream=None) -> None:
    _check(lib().gemm_bt(_ptr(A), _ptr(B), _ptr(out), _ptr(workspace), workspace_bytes, M, N, K,
                         splits, k_per_split, dtype_code(dtype), fused, _stream(stream)), "gemm_bt")


def gemm_bt_noalloc(A, B, out, M, N, K, splits, k_per_split, dtype, fused=0, stream=None) -> None:
    """gemm_bt without a workspace argument, for callers that cannot allocate:
    the library's own device scratch array serves instead (see splitk.h)."""
    _check(lib().gemm_bt_noalloc(_ptr(A), _ptr(B), _ptr(out), M, N, K, splits, k_per_split,
                                 dtype_code(dtype), fused, _stream(stream)), "gemm_bt_noalloc")


def gemm_bt_host_staging_bytes(count, M, N, K, splits, k_per_split, dtype) -> int:
    return lib().gemm_bt_host_staging_bytes(count, M, N, K, splits, k_per_split, dtype_code(dtype))


def pointer_array(items):
    """A C array of device pointers (tensors or integer addresses); keep it
    alive for the duration of the call that receives it."""
    arr = (ctypes.c_void_p * max(len(items), 1))()
    for i, x in enumerate(items):
        arr[i] = _ptr(x)
    return arr


def gemm_bt_host_batch(A_host, B, out_host, count, staging, staging_bytes, M, N, K, splits, k_per_split,
                       dtype, fused=0, ops_per_copy=0, stream=None) -> None:
    """A_host and out_host: host tensors (pinned for overlap) or addresses; B:
    a sequence of `count` device weights, or a prebuilt pointer_array()."""
    arr = B if isinstance(B, ctypes.Array) else pointer_array(B)
    _check(lib().gemm_bt_host_batch(_ptr(A_host), ctypes.cast(arr, ctypes.c_void_p), _ptr(out_host), count,
                                    _ptr(staging), staging_bytes, M, N, K, splits, k_per_split,
                                    dtype_code(dtype), fused, ops_per_copy, _stream(stream)),
           "gemm_bt_host_batch")


def gemm_bt_batch(A, B, out, count, workspace, workspace_bytes, M, N, K, splits, k_per_split, dtype, fused=0,
                  stream=None) -> None:
    """`count` operations out[i] = gemm_bt(A[i], B[i]) of one shape; A, B and
    out: sequences of device tensors (or addresses), or prebuilt
    pointer_array()s."""
    arrs = [x if isinstance(x, ctypes.Array) else pointer_array(x) for x in (A, B, out)]
    _check(lib().gemm_bt_batch(*(ctypes.cast(a, ctypes.c_void_p) for a in arrs), count, _ptr(workspace),
                               workspace_bytes, M, N, K, splits, k_per_split, dtype_code(dtype), fused,
                               _stream(stream)), "gemm_bt_batch")


SPLIT_CANDIDATES = (1, 2, 4, 8, 16)


def splitk_choose_splits(M, N, K, dtype, fused=0) -> tuple[int, int, dict]:
    """(splits, k_per_split, {candidate: model microseconds or None}) from the
    library's cost model."""
    s, k = ctypes.c_int64(), ctypes.c_int64()
    t = (ctypes.c_double * len(SPLIT_CANDIDATES))()
    _check(lib().splitk_choose_splits(M, N, K, dtype_code(dtype), fused, ctypes.byref(s), ctypes.byref(k), t),
           "splitk_choose_splits")
    return s.value, k.value, {c: (None if t[i] < 0 else float(t[i])) for i, c in enumerate(SPLIT_CANDIDATES)}


def splitk_autotune_splits(A, B, out, workspace, workspace_bytes, M, N, K, dtype, fused=0, reps=20,
                           stream=None) -> tuple[int, int, dict]:
    """(splits, k_per_split, {candidate: us per call or None}) measured on the device."""
    s, k = ctypes.c_int64(), ctypes.c_int64()
    us = (ctypes.c_float * len(SPLIT_CANDIDATES))()
    _check(lib().splitk_autotune_splits(_ptr(A), _ptr(B), _ptr(out), _ptr(workspace), workspace_bytes, M, N, K,
                                        dtype_code(dtype), fused, reps, _stream(stream), ctypes.byref(s),
                                        ctypes.byref(k), us), "splitk_autotune_splits")
    return s.value, k.value, {c: (None if us[i] < 0 else float(us[i])) for i, c in enumerate(SPLIT_CANDIDATES)}


def splitk_get_device_status(stream=None) -> int:
    """Synchronises the stream, then reads and clears the device status word."""
    return lib().splitk_get_device_status(_stream(stream))


def splitk_set_tile_override(bn: int = 0, chunks: int = 0, kblocks_per_stage: int = 0) -> None:
    _check(lib().splitk_set_tile_override(bn, chunks, kblocks_per_stage), "splitk_set_tile_override")


def splitk_describe_launch(M, N, K, splits, k_per_split, dtype, fused=0) -> dict:
    info = (ctypes.c_int * 26)()
    _check(lib().splitk_describe_launch(M, N, K, splits, k_per_split, dtype_code(dtype), fused,
                                        ctypes.addressof(info)), "splitk_describe_launch")
    keys = ("path", "bn", "chunks", "chunk_len", "stages", "cluster", "grid_x", "grid_y",
            "grid_z", "smem_bytes", "fused_in_kernel", "kernels_per_call", "kblocks_per_stage",
            "three_d", "split_sum", "prefetchers", "rows_first", "tile_m",
            "compact", "compact_stages", "compact_kblocks_per_stage", "compact_smem_bytes",
            "compact_chunks_per_block", "compact_cluster", "compact_grid_z", "compact_bn")
    return dict(zip(keys, list(info)))


def splitk_selftest_bounded_wait(limit_ns: int = 1_000_000, stream=None) -> int:
    return lib().splitk_selftest_bounded_wait(limit_ns, _stream(stream))


def splitk_set_overlap(mode=2) -> None:
    """Consecutive independent calls inside graph captures, for later
    captures of the whole process: 2 (or True, the default) overlap and group
    them, 1 overlap only, 0 (or False) neither."""
    if isinstance(mode, bool):
        mode = 2 if mode else 0
    _check(lib().splitk_set_overlap(int(mode)), "splitk_set_overlap")


def splitk_last_launch() -> dict:
    """What the calling thread's most recent tensor-core launch did."""
    info = (ctypes.c_int * 11)()
    _check(lib().splitk_last_launch(ctypes.addressof(info)), "splitk_last_launch")
    keys = ("overlap", "compact", "capturing", "bn", "chunks", "stages", "kblocks_per_stage", "smem_bytes",
            "chunks_per_block", "cluster", "group")
    return dict(zip(keys, list(info)))


def splitk_selftest_kernel_timeout(A, B, out, M, N, K, splits, k_per_split, dtype, stream=None) -> int:
    """One fused launch whose wait for the final accumulator gives up at once
    (the kernel's own time-out path); returns the device status it leaves
    (ERR_DEVICE_TIMEOUT expected).  Never raises."""
    return lib().splitk_selftest_kernel_timeout(_ptr(A), _ptr(B), _ptr(out), M, N, K, splits, k_per_split,
                                                dtype_code(dtype), _stream(stream))
