"""fp64 CPU oracle for the KDA operator -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes anything here.

Contents:
  * ``kda_oracle.c`` -- the token-by-token fp64 recurrence (the oracle proper),
    built with gcc into ``_build/libkda_oracle.so`` and called through ctypes.
  * ``chunked.py``   -- the chunk-parallel form of the same recurrence, written
    out in numpy fp64 step by step; used only to pin the recurrence.
  * ``exact.py``     -- the recurrence in exact rational arithmetic for tiny
    inputs (Python ``fractions``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (plain C11, -O2, no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def _f64(x) -> np.ndarray:
    """Exact upcast to a C-contiguous float64 numpy array (bf16/fp32 values are exact in fp64)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _per_channel(la: np.ndarray, dk: int) -> np.ndarray:
    """A scalar gate (log_alpha [T, H], one per token and head: the Gated
    DeltaNet gate, "Kimi Delta Attention" deep dive, section 03) is the
    per-channel gate with the same value in every key channel; the C oracle
    takes the per-channel form, so the scalar is repeated over d_k."""
    if la.ndim == 2:
        return np.ascontiguousarray(np.repeat(la[:, :, None], dk, axis=2))
    return la


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


class Oracle:
    """ctypes front end of one build of ``kda_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i32 = ctypes.c_int32
        lib.kda_oracle_prefill.argtypes = [i32, i32, i32, i32, ip, dp, dp, dp, dp, dp, dp, dp, dp,
                                           i32, i32, i32]
        lib.kda_oracle_prefill.restype = ctypes.c_int
        lib.kda_oracle_decode_step.argtypes = [i32, i32, i32, i32, dp, dp, dp, dp, dp, dp, dp, i32]
        lib.kda_oracle_decode_step.restype = ctypes.c_int
        lib.kda_oracle_backward.argtypes = [i32, i32, i32, i32, ip] + [dp] * 14 + [i32]
        lib.kda_oracle_backward.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def prefill(self, q, k, v, log_alpha, beta, cu_seqlens=None, initial_state=None,
                cols: Optional[tuple] = None, threads: Optional[int] = None):
        """fp64 prefill.  Returns (out [T,H,d_v], final_state [N,H,d_k,d_v]) as float64 numpy.

        ``cols=(j0, j1)`` computes only those columns of out / final_state (the
        others stay NaN): columns of the state are independent, so this is the
        exact result for those columns at a fraction of the cost.
        """
        q, k, v, la, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
        T, H, dk = q.shape
        dv = v.shape[2]
        la = _per_channel(la, dk)
        if cu_seqlens is None:
            cu = np.array([0, T], dtype=np.int32)
        else:
            if hasattr(cu_seqlens, "cpu"):
                cu_seqlens = cu_seqlens.cpu().numpy()
            cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = len(cu) - 1
        s0 = None if initial_state is None else _f64(initial_state).reshape(N, H, dk, dv)
        out = np.full((T, H, dv), np.nan)
        sf = np.full((N, H, dk, dv), np.nan)
        j0, j1 = (0, dv) if cols is None else cols
        rc = self.lib.kda_oracle_prefill(N, H, dk, dv, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                         _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(s0),
                                         _ptr(out), _ptr(sf), j0, j1, threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"kda_oracle_prefill failed: {rc}")
        return out, sf

    def backward(self, q, k, v, log_alpha, beta, cu_seqlens=None, initial_state=None, dout=None,
                 dfinal=None, threads: Optional[int] = None):
        """fp64 gradients of a scalar loss through the prefill, given its
        gradients ``dout`` [T,H,d_v] and ``dfinal`` [N,H,d_k,d_v] (None: zero).

        Returns a dict of float64 arrays: dq, dk, dv, dlog_alpha (the shape of
        ``log_alpha``: a scalar gate [T,H] gets the sum over channels), dbeta,
        dinitial_state."""
        q, k, v, la, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
        T, H, dk = q.shape
        dv = v.shape[2]
        scalar_gate = la.ndim == 2
        la = _per_channel(la, dk)
        if cu_seqlens is None:
            cu = np.array([0, T], dtype=np.int32)
        else:
            if hasattr(cu_seqlens, "cpu"):
                cu_seqlens = cu_seqlens.cpu().numpy()
            cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = len(cu) - 1
        s0 = None if initial_state is None else _f64(initial_state).reshape(N, H, dk, dv)
        do = _f64(dout).reshape(T, H, dv)
        dfin = None if dfinal is None else _f64(dfinal).reshape(N, H, dk, dv)
        g = {"dq": np.zeros((T, H, dk)), "dk": np.zeros((T, H, dk)), "dv": np.zeros((T, H, dv)),
             "dlog_alpha": np.zeros((T, H, dk)), "dbeta": np.zeros((T, H)),
             "dinitial_state": np.zeros((N, H, dk, dv))}
        rc = self.lib.kda_oracle_backward(N, H, dk, dv, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                          _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), _ptr(s0), _ptr(do),
                                          _ptr(dfin), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                                          _ptr(g["dlog_alpha"]), _ptr(g["dbeta"]), _ptr(g["dinitial_state"]),
                                          threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"kda_oracle_backward failed: {rc}")
        if scalar_gate:
            g["dlog_alpha"] = g["dlog_alpha"].sum(axis=2)
        return g

    def decode_step(self, q, k, v, log_alpha, beta, state, threads: Optional[int] = None):
        """fp64 decode step.  Inputs [N,H,*]; returns (out [N,H,d_v], new_state)."""
        q, k, v, la, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
        N, H, dk = q.shape
        dv = v.shape[2]
        la = _per_channel(la, dk)
        s = _f64(state).reshape(N, H, dk, dv).copy()
        out = np.full((N, H, dv), np.nan)
        rc = self.lib.kda_oracle_decode_step(N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(la),
                                             _ptr(b), _ptr(s), _ptr(out), threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"kda_oracle_decode_step failed: {rc}")
        return out, s


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def prefill(*args, **kwargs):
    """fp64 prefill with the default oracle build (see ``Oracle.prefill``)."""
    return default().prefill(*args, **kwargs)


def decode_step(*args, **kwargs):
    """fp64 decode step with the default oracle build (see ``Oracle.decode_step``)."""
    return default().decode_step(*args, **kwargs)


def backward(*args, **kwargs):
    """fp64 prefill gradients with the default oracle build (see ``Oracle.backward``)."""
    return default().backward(*args, **kwargs)
