"""Seeded, counter-based synthetic inputs for the KDA operator.

This module is shared by the CUDA path's tests/benchmark and by the fp64
oracle's tests, as *input data only*.  It holds none of the KDA arithmetic:
it draws random numbers, normalises the drawn q/k vectors, applies the
sigmoid that turns a normal draw into beta, and rounds to the storage dtype.
These are the input distributions of the five synthetic workloads (the
gates are passed to the operator already in their final form: beta after
the sigmoid, alpha as log_alpha).

Random numbers come from one counter-based generator: value i of stream s
under seed r is ``splitmix64(key(r, s) + i)`` where ``key`` is itself built
from splitmix64.  splitmix64 is Steele, Lea & Flood, "Fast splittable
pseudorandom number generators" (OOPSLA 2014).  Uniforms take the top 53
bits; normals use the Box-Muller transform on two uniforms drawn from
counters 2i and 2i+1.  Everything is computed in float64 with torch on the
requested device and then rounded once (round-to-nearest-even) to the
storage dtype, so any slice of a tensor can be regenerated on its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

_MASK64 = (1 << 64) - 1


def _to_signed(x: int) -> int:
    x &= _MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


_GAMMA = 0x9E3779B97F4A7C15
_MUL1 = 0xBF58476D1CE4E5B9
_MUL2 = 0x94D049BB133111EB


def splitmix64_int(x: int) -> int:
    """splitmix64 finaliser on a Python int (exact 64-bit unsigned arithmetic)."""
    z = (x + _GAMMA) & _MASK64
    z = ((z ^ (z >> 30)) * _MUL1) & _MASK64
    z = ((z ^ (z >> 27)) * _MUL2) & _MASK64
    return z ^ (z >> 31)


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor holding 64-bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def splitmix64(x: torch.Tensor) -> torch.Tensor:
    """splitmix64 on an int64 tensor (two's-complement wrap-around arithmetic)."""
    z = x + _to_signed(_GAMMA)
    z = (z ^ _srl(z, 30)) * _to_signed(_MUL1)
    z = (z ^ _srl(z, 27)) * _to_signed(_MUL2)
    return z ^ _srl(z, 31)


# Stream identifiers: one per drawn tensor.  Decode step s (0-based) uses
# stream id + 16 * (s + 1) so that every step draws fresh values.
STREAMS = {"lengths": 1, "q": 2, "k": 3, "v": 4, "beta": 5, "log_alpha": 6, "state": 7}


def stream_key(seed: int, stream: int) -> int:
    return splitmix64_int(splitmix64_int(seed) ^ (stream * 0x100000001B3))


def raw_bits(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """64-bit words ``start .. start+count-1`` of stream ``stream`` (int64 tensor)."""
    key = _to_signed(stream_key(seed, stream))
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    return splitmix64(idx + key)


def uniform(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """float64 uniforms in [0, 1) from the top 53 bits of each word."""
    return _srl(raw_bits(seed, stream, start, count, device), 11).to(torch.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """float64 standard normals (Box-Muller on words 2i and 2i+1)."""
    u = uniform(seed, stream, 2 * start, 2 * count, device).view(count, 2)
    r = torch.sqrt(-2.0 * torch.log1p(-u[:, 0]))   # 1 - u1 lies in (0, 1]
    return r * torch.cos((2.0 * math.pi) * u[:, 1])


# ----------------------------------------------------------------------------
# Workload recipes
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    """Shape and value distributions of one synthetic workload."""
    name: str
    seed: int
    num_heads: int
    d_k: int
    d_v: int
    dtype: str                      # "f32" or "bf16": storage dtype of q,k,v,beta,log_alpha,out
    seqlens: list = field(default_factory=list)   # prefill: per-sequence lengths
    la_lo: float = 0.0005           # log_alpha = -U(la_lo, la_hi)
    la_hi: float = 0.1
    state_std: Optional[float] = 0.02   # None: zero initial state
    decode_seqs: int = 0            # decode workloads: sequences per step
    decode_steps: int = 0
    gate: str = "channel"           # "channel": log_alpha [.., H, d_k]; "scalar": one per (token, head) [.., H]

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens) if self.decode_seqs == 0 else self.decode_seqs

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def varlen_lengths(seed: int, n: int, lo: int, hi: int) -> list:
    """n integer lengths uniform on [lo, hi] (inclusive)."""
    u = uniform(seed, STREAMS["lengths"], 0, n)
    return [int(lo + min(int(x * (hi - lo + 1)), hi - lo)) for x in u.tolist()]


def workload(index: int) -> Workload:
    """The five synthetic workloads of the KDA hot path, by index.

    0: one sequence T=256, H=2, d=64, fp32, zero initial state,
       log_alpha = -U(0.001, 0.2).
    1: one sequence T=4096, H=16, d=128, bf16 inputs, initial state ~N(0, 0.02^2),
       log_alpha = -U(0.0005, 0.1).
    2: varlen, 8 sequences with lengths U[512, 16384] drawn from the seed,
       H=32, d=128, bf16, distributions as workload 1.
    3: decode, 256 sequences x 1 token, H=32, d=128, fp32 state ~N(0, 0.02^2),
       bf16 inputs as workload 1, 64 consecutive steps.
    4: one sequence T=2^20, H=16, d=128, bf16, log_alpha = -U(0.0001, 0.05),
       initial state ~N(0, 0.02^2); its final state feeds one decode step.
    """
    if index == 0:
        return Workload("single_T256_H2_d64_f32", 0, 2, 64, 64, "f32", [256],
                        la_lo=0.001, la_hi=0.2, state_std=None)
    if index == 1:
        return Workload("prefill_T4096_H16_d128_bf16", 1, 16, 128, 128, "bf16", [4096])
    if index == 2:
        return Workload("varlen8_U512_16384_H32_d128_bf16", 2, 32, 128, 128, "bf16",
                        varlen_lengths(2, 8, 512, 16384))
    if index == 3:
        return Workload("decode_N256_H32_d128_bf16x64", 3, 32, 128, 128, "bf16", [],
                        decode_seqs=256, decode_steps=64)
    if index == 4:
        return Workload("prefill_T1048576_H16_d128_bf16", 4, 16, 128, 128, "bf16", [1 << 20],
                        la_lo=0.0001, la_hi=0.05)
    raise ValueError(f"no workload {index}")


def custom(seed: int, seqlens, num_heads: int, d: int, dtype: str = "bf16",
           la_lo: float = 0.0005, la_hi: float = 0.1, state_std: Optional[float] = 0.02,
           d_v: Optional[int] = None, gate: str = "channel", decode_seqs: int = 0) -> Workload:
    """A workload with the distributions of workload 1 and a caller-chosen shape.
    ``gate="scalar"`` draws one log_alpha per (token, head) (the Gated DeltaNet
    gate) instead of one per key channel."""
    if gate not in ("channel", "scalar"):
        raise ValueError(f"gate must be 'channel' or 'scalar', not {gate!r}")
    return Workload(f"custom_s{seed}" + ("_scalar" if gate == "scalar" else ""), seed, num_heads, d,
                    d if d_v is None else d_v, dtype, list(seqlens), la_lo=la_lo, la_hi=la_hi,
                    state_std=state_std, gate=gate, decode_seqs=decode_seqs)


def _round(x64: torch.Tensor, dtype) -> torch.Tensor:
    return x64.to(dtype)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


def _draw_tokens(w: Workload, stream_offset: int, t0: int, t1: int, device):
    """q, k, v, beta, log_alpha for tokens [t0, t1) of the packed batch."""
    H, dk, dv = w.num_heads, w.d_k, w.d_v
    n = t1 - t0
    st = lambda name: STREAMS[name] + stream_offset
    q = normal(w.seed, st("q"), t0 * H * dk, n * H * dk, device).view(n, H, dk)
    k = normal(w.seed, st("k"), t0 * H * dk, n * H * dk, device).view(n, H, dk)
    v = normal(w.seed, st("v"), t0 * H * dv, n * H * dv, device).view(n, H, dv)
    b = normal(w.seed, st("beta"), t0 * H, n * H, device).view(n, H)
    if w.gate == "scalar":
        u = uniform(w.seed, st("log_alpha"), t0 * H, n * H, device).view(n, H)
    else:
        u = uniform(w.seed, st("log_alpha"), t0 * H * dk, n * H * dk, device).view(n, H, dk)
    q = _unit_rows(q) * (1.0 / math.sqrt(dk))
    k = _unit_rows(k)
    beta = torch.sigmoid(b)
    log_alpha = -(w.la_lo + (w.la_hi - w.la_lo) * u)
    dt = w.torch_dtype
    return {"q": _round(q, dt), "k": _round(k, dt), "v": _round(v, dt),
            "beta": _round(beta, dt), "log_alpha": _round(log_alpha, dt)}


def prefill_inputs(w: Workload, device="cpu", t_range=None, block_tokens: int = 1 << 15):
    """Inputs of a prefill workload, in the storage dtype, on ``device``.

    Layouts (row-major): q, k, log_alpha [T, H, d_k]; v [T, H, d_v]; beta [T, H];
    cu_seqlens int32 [N+1]; initial_state fp32 [N, H, d_k, d_v] (None for a
    zero state).  ``t_range=(t0, t1)`` generates only those packed tokens
    (cu_seqlens and the state are still returned whole).
    """
    T = w.total_tokens
    t0, t1 = (0, T) if t_range is None else t_range
    parts = {name: [] for name in ("q", "k", "v", "beta", "log_alpha")}
    for a in range(t0, t1, block_tokens):
        b = min(t1, a + block_tokens)
        d = _draw_tokens(w, 0, a, b, device)
        for name in parts:
            parts[name].append(d[name])
    out = {}
    for name, lst in parts.items():
        if lst:
            out[name] = torch.cat(lst) if len(lst) > 1 else lst[0]
        else:
            shape = {"q": (0, w.num_heads, w.d_k), "k": (0, w.num_heads, w.d_k),
                     "log_alpha": (0, w.num_heads) if w.gate == "scalar" else (0, w.num_heads, w.d_k),
                     "v": (0, w.num_heads, w.d_v),
                     "beta": (0, w.num_heads)}[name]
            out[name] = torch.empty(shape, dtype=w.torch_dtype, device=device)
    cu = [0]
    for L in w.seqlens:
        cu.append(cu[-1] + int(L))
    out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32, device=device)
    out["initial_state"] = initial_state(w, len(w.seqlens), device)
    return out


def initial_state(w: Workload, num_seqs: int, device="cpu"):
    """fp32 [N, H, d_k, d_v] ~ N(0, state_std^2), or None for a zero state."""
    if w.state_std is None:
        return None
    n = num_seqs * w.num_heads * w.d_k * w.d_v
    s = normal(w.seed, STREAMS["state"], 0, n, device) * w.state_std
    return s.to(torch.float32).view(num_seqs, w.num_heads, w.d_k, w.d_v)


def decode_inputs(w: Workload, step: int, device="cpu"):
    """Fresh q, k, v, beta, log_alpha for decode step ``step`` (one token per sequence)."""
    return _draw_tokens(w, 16 * (step + 1), 0, w.decode_seqs, device)
