"""ctypes binding of libkda.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.environ.get("KDA_LIBRARY", os.path.join(_HERE, "_build", "libkda.so"))

KDA_OK, KDA_ERR_INVALID_ARGUMENT, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA = 0, 1, 2, 3
KDA_ERR_TIMEOUT, KDA_ERR_BAD_SEQLENS, KDA_ERR_WORKSPACE, KDA_ERR_BAD_SNAPSHOT = 4, 5, 6, 7
KDA_F32, KDA_BF16 = 0, 1
KDA_FLAG_CUDA_CORE_PREFILL = 1
KDA_FLAG_SCALAR_GATE = 2

EXPORTS = ("kda_prefill_workspace_bytes", "kda_prefill", "kda_decode_step", "kda_get_device_status",
           "kda_status_string", "kda_last_cuda_error", "kda_version", "kda_prefill_noalloc",
           "kda_selftest_wait_timeout", "kda_prefill_snapshots", "kda_backward_workspace_bytes",
           "kda_prefill_backward")
KDA_PREFILL_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class KdaDesc(ctypes.Structure):
    """Mirror of ``kda_desc`` in include/kda.h."""
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("phase_events", ctypes.c_void_p)]


class KdaError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        extra = ""
        if status == KDA_ERR_CUDA:
            extra = f" (cudaError {lib.kda_last_cuda_error()})"
        super().__init__(f"{call} failed: {kda_status_string(status)}{extra}")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libkda.so not built at {_LIB_PATH}: run "
                          f"`python -c 'import __graft_entry__ as g; g.build()'` first")
    L = ctypes.CDLL(_LIB_PATH)
    vp, D = ctypes.c_void_p, ctypes.POINTER(KdaDesc)
    L.kda_prefill_workspace_bytes.argtypes = [D]
    L.kda_prefill_workspace_bytes.restype = ctypes.c_size_t
    L.kda_prefill.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.kda_prefill.restype = ctypes.c_int
    L.kda_prefill_snapshots.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp]
    L.kda_prefill_snapshots.restype = ctypes.c_int
    L.kda_backward_workspace_bytes.argtypes = [D]
    L.kda_backward_workspace_bytes.restype = ctypes.c_size_t
    L.kda_prefill_backward.argtypes = [D] + [vp] * 16
    L.kda_prefill_backward.restype = ctypes.c_int
    L.kda_prefill_noalloc.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.kda_prefill_noalloc.restype = ctypes.c_int
    L.kda_selftest_wait_timeout.argtypes = [D, ctypes.c_int64, vp]
    L.kda_selftest_wait_timeout.restype = ctypes.c_int
    L.kda_decode_step.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp]
    L.kda_decode_step.restype = ctypes.c_int
    L.kda_get_device_status.argtypes = [D, vp]
    L.kda_get_device_status.restype = ctypes.c_int
    L.kda_status_string.argtypes = [ctypes.c_int]
    L.kda_status_string.restype = ctypes.c_char_p
    L.kda_last_cuda_error.argtypes = []
    L.kda_last_cuda_error.restype = ctypes.c_int
    L.kda_version.argtypes = []
    L.kda_version.restype = ctypes.c_int
    return L


lib = _load()


def prefill_kernel_files(dtype: str, d: int, flags: int = 0):
    """Source files of the two prefill kernels the library runs for a dtype and head size."""
    if dtype == "bf16" and d == 128 and not (flags & KDA_FLAG_CUDA_CORE_PREFILL):
        files = ["kda_prefill_tc.cu", "kda_tc_record.cuh", "kda_sm100.cuh", "kda_common.cuh"]
    else:
        files = ["kda_prefill_simt.cu", "kda_common.cuh"]
    return {"intra": files, "chain": files}


def library_path() -> str:
    return os.path.realpath(_LIB_PATH)


def exported_symbols():
    """Names of the C ABI entry points found in the loaded library."""
    return [n for n in EXPORTS if hasattr(lib, n)]


def kda_status_string(status: int) -> str:
    return lib.kda_status_string(int(status)).decode()


def kda_version() -> int:
    return lib.kda_version()


_DTYPES = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}


def make_desc(num_seqs: int, num_heads: int, d_k: int, d_v: int, total_tokens: int, dtype,
              workspace: Optional[torch.Tensor] = None, flags: int = 0) -> KdaDesc:
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    d = KdaDesc(num_seqs, num_heads, d_k, d_v, total_tokens, dt, flags, None, 0, None)
    if workspace is not None:
        d.workspace = workspace.data_ptr()
        d.workspace_bytes = workspace.numel() * workspace.element_size()
    return d


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def kda_prefill_workspace_bytes(desc: KdaDesc) -> int:
    return lib.kda_prefill_workspace_bytes(ctypes.byref(desc))


def kda_prefill(desc: KdaDesc, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state,
                stream=None) -> int:
    """Raw C call: every tensor argument is passed as its data pointer (or NULL)."""
    return lib.kda_prefill(ctypes.byref(desc), _p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
                           _p(cu_seqlens), _p(initial_state), _p(out), _p(final_state), _stream(stream))


def kda_prefill_snapshots(desc: KdaDesc, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state,
                          num_snapshots: int, snapshot_at, snapshots, stream=None) -> int:
    """Raw C call of the prefill with state snapshots (see include/kda.h)."""
    return lib.kda_prefill_snapshots(ctypes.byref(desc), _p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
                                     _p(cu_seqlens), _p(initial_state), _p(out), _p(final_state),
                                     int(num_snapshots), _p(snapshot_at), _p(snapshots), _stream(stream))


def kda_backward_workspace_bytes(desc: KdaDesc) -> int:
    return lib.kda_backward_workspace_bytes(ctypes.byref(desc))


def kda_prefill_backward(desc: KdaDesc, q, k, v, log_alpha, beta, cu_seqlens, initial_state, d_out, d_final_state,
                         dq, dk, dv, dlog_alpha, dbeta, d_initial_state, stream=None) -> int:
    """Raw C call of the prefill's reverse mode (see include/kda.h)."""
    return lib.kda_prefill_backward(ctypes.byref(desc), _p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
                                    _p(cu_seqlens), _p(initial_state), _p(d_out), _p(d_final_state), _p(dq),
                                    _p(dk), _p(dv), _p(dlog_alpha), _p(dbeta), _p(d_initial_state),
                                    _stream(stream))


def prefill_backward(q, k, v, log_alpha, beta, cu_seqlens=None, initial_state=None, *, d_out,
                     d_final_state=None, want_initial_grad: bool = True, workspace=None, stream=None,
                     flags: int = 0):
    """Gradients of a loss through kda_prefill (fp32 tensors), given d_out and
    optionally d_final_state.  A 2-D ``log_alpha`` selects the scalar gate;
    ``flags=KDA_FLAG_CUDA_CORE_PREFILL`` selects the fp32 CUDA-core backward
    where the tensor-core one would run (bf16, head size 128).
    Returns a dict: dq, dk, dv, dlog_alpha, dbeta, d_initial_state (or None)."""
    T, H, dk_ = q.shape
    dv_ = v.shape[2]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("log_alpha", log_alpha), ("beta", beta), ("d_out", d_out)):
        _check(t, name)
    if log_alpha.dim() == 2:
        flags |= KDA_FLAG_SCALAR_GATE
    f32 = dict(dtype=torch.float32, device=q.device)
    g = {"dq": torch.empty((T, H, dk_), **f32), "dk": torch.empty((T, H, dk_), **f32),
         "dv": torch.empty((T, H, dv_), **f32), "dlog_alpha": torch.empty(tuple(log_alpha.shape), **f32),
         "dbeta": torch.empty((T, H), **f32),
         "d_initial_state": torch.empty((N, H, dk_, dv_), **f32) if want_initial_grad else None}
    desc = make_desc(N, H, dk_, dv_, T, q.dtype, flags=flags)
    if workspace is None:
        nbytes = kda_backward_workspace_bytes(desc)
        if nbytes == 0:
            raise KdaError("kda_backward_workspace_bytes", KDA_ERR_UNSUPPORTED)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    desc.workspace = workspace.data_ptr()
    desc.workspace_bytes = workspace.numel()
    rc = kda_prefill_backward(desc, q, k, v, log_alpha, beta, cu_seqlens, initial_state, d_out, d_final_state,
                              g["dq"], g["dk"], g["dv"], g["dlog_alpha"], g["dbeta"], g["d_initial_state"], stream)
    if rc != KDA_OK:
        raise KdaError("kda_prefill_backward", rc)
    return g


def kda_prefill_noalloc(desc: KdaDesc, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state,
                        stream=None) -> int:
    """Raw C call of the no-workspace prefill (the library's fixed scratch area)."""
    return lib.kda_prefill_noalloc(ctypes.byref(desc), _p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
                                   _p(cu_seqlens), _p(initial_state), _p(out), _p(final_state), _stream(stream))


def kda_selftest_wait_timeout(desc: KdaDesc, timeout_ns: int, stream=None) -> int:
    """Run the bounded-wait failure path on the GPU (see include/kda.h)."""
    return lib.kda_selftest_wait_timeout(ctypes.byref(desc), int(timeout_ns), _stream(stream))


def kda_decode_step(desc: KdaDesc, q, k, v, log_alpha, beta, state_inout, out, stream=None) -> int:
    return lib.kda_decode_step(ctypes.byref(desc), _p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
                               _p(state_inout), _p(out), _stream(stream))


def kda_get_device_status(desc: KdaDesc, stream=None) -> int:
    return lib.kda_get_device_status(ctypes.byref(desc), _stream(stream))


def _check(t: torch.Tensor, name: str):
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def prefill(q, k, v, log_alpha, beta, cu_seqlens=None, initial_state=None, *, out=None,
            final_state=None, workspace=None, stream=None, want_final_state: bool = True, flags: int = 0,
            snapshot_at=None, snapshots=None):
    """Chunk-parallel prefill (see kda_prefill in include/kda.h).

    Allocates ``out``, ``final_state`` and the workspace with torch when they
    are not given.  A 2-D ``log_alpha`` [T, H] selects the scalar gate
    (KDA_FLAG_SCALAR_GATE).  Returns (out, final_state, workspace).

    ``snapshot_at`` (int32 [M, 2] CUDA tensor of (sequence, prefix length)
    pairs) also saves the state after each of those prefixes into
    ``snapshots`` [M, H, d_k, d_v] (allocated if not given) through
    kda_prefill_snapshots; the call then returns (out, final_state, workspace,
    snapshots)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    if log_alpha.dim() == 2:
        flags |= KDA_FLAG_SCALAR_GATE
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    for name, t in (("q", q), ("k", k), ("v", v), ("log_alpha", log_alpha), ("beta", beta)):
        _check(t, name)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None and want_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    desc = make_desc(N, H, dk, dv, T, q.dtype, flags=flags)
    if workspace is None:
        nbytes = kda_prefill_workspace_bytes(desc)
        if nbytes == 0:
            raise KdaError("kda_prefill_workspace_bytes", KDA_ERR_UNSUPPORTED)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    desc.workspace = workspace.data_ptr()
    desc.workspace_bytes = workspace.numel()
    if snapshot_at is None:
        rc = kda_prefill(desc, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state, stream)
        if rc != KDA_OK:
            raise KdaError("kda_prefill", rc)
        return out, final_state, workspace
    _check(snapshot_at, "snapshot_at")
    if snapshot_at.dtype != torch.int32 or snapshot_at.dim() != 2 or snapshot_at.shape[1] != 2:
        raise ValueError("snapshot_at must be an int32 [M, 2] tensor of (sequence, prefix length)")
    M = snapshot_at.shape[0]
    if snapshots is None:
        snapshots = torch.empty((M, H, dk, dv), dtype=torch.float32, device=q.device)
    rc = kda_prefill_snapshots(desc, q, k, v, log_alpha, beta, cu_seqlens, initial_state, out, final_state,
                               M, snapshot_at, snapshots, stream)
    if rc != KDA_OK:
        raise KdaError("kda_prefill_snapshots", rc)
    return out, final_state, workspace, snapshots


def decode_step(q, k, v, log_alpha, beta, state, *, out=None, stream=None):
    """One decode step, ``state`` [N,H,d_k,d_v] fp32 updated in place.  A 2-D
    ``log_alpha`` [N, H] selects the scalar gate.  Returns out."""
    N, H, dk = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    desc = make_desc(N, H, dk, dv, N, q.dtype, flags=KDA_FLAG_SCALAR_GATE if log_alpha.dim() == 2 else 0)
    rc = kda_decode_step(desc, q, k, v, log_alpha, beta, state, out, stream)
    if rc != KDA_OK:
        raise KdaError("kda_decode_step", rc)
    return out
