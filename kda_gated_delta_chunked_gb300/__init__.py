"""GB300 (sm_103a) Kimi Delta Attention hot path: chunk-parallel varlen prefill
and the one-token recurrent decode step.

The compute runs in the hand-written CUDA kernels of ``libkda.so`` (C ABI in
``include/kda.h``).  This package is a thin ctypes binding with the same entry
point names; it only marshals torch tensors into pointers and sizes.  If the
library has not been built, importing the package raises -- there is no
fallback implementation.
"""
from ._binding import (  # noqa: F401
    KDA_OK, KDA_ERR_INVALID_ARGUMENT, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT,
    KDA_ERR_BAD_SEQLENS, KDA_ERR_WORKSPACE, KDA_ERR_BAD_SNAPSHOT, KDA_F32, KDA_BF16, KDA_FLAG_CUDA_CORE_PREFILL, KDA_FLAG_SCALAR_GATE, KdaDesc,
    KdaError, prefill_kernel_files,
    library_path, lib, exported_symbols,
    kda_prefill_workspace_bytes, kda_prefill, kda_decode_step, kda_get_device_status,
    kda_status_string, kda_version, make_desc, prefill, decode_step, kda_prefill_noalloc,
    KDA_PREFILL_NOALLOC_SCRATCH_BYTES, kda_selftest_wait_timeout, kda_prefill_snapshots,
    kda_backward_workspace_bytes, kda_prefill_backward, prefill_backward,
)
