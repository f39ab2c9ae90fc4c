"""split_bf16_gemm_gb300 -- split-K GEMM with prepared, transposed weights on GB300.

A[M,K] (row-major) times the prepared weight B[N,K] (row-major, the transpose
of a [K,N] weight), split along K into F32 partials[splits,M,N], then summed
over splits into the F32 [M,N] output.  The compute runs in libsplitk, a C-ABI
CUDA library for sm_103a (tcgen05 tensor cores: native BF16/F16, 3xTF32 for
F32); this package is its build step and a thin ctypes binding.
"""
from ._build import LIB_PATH, build  # noqa: F401
from .binding import (  # noqa: F401
    BF16, F16, F32, SplitKError, dtype_code, gemm_bt, gemm_bt_batch, gemm_bt_host_batch, gemm_bt_host_staging_bytes,
    gemm_bt_noalloc, gemm_bt_workspace_bytes, gemm_bt_workspace_init, gemm_kn, gemm_splitk_kn, pointer_array,
    gemm_splitk_bt,
    lib, splitk_check_geometry, splitk_describe_launch, splitk_get_device_status, splitk_reduce,
    splitk_autotune_splits, splitk_choose_splits, splitk_last_error, splitk_last_launch, splitk_prepare_bt,
    splitk_selftest_bounded_wait, splitk_selftest_kernel_timeout, splitk_set_overlap, splitk_set_tile_override,
    splitk_status_string,
    status_string,
)
