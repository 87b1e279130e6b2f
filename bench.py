#!/usr/bin/env python
"""Benchmark of the GB300 KDA hot path.

One step = one pass of the whole hot path over one batch of synthetic input:
the chunk-parallel prefill of the 1M-token workload (T = 2^20, H = 16,
d_k = d_v = 128, bf16 inputs, fp32 state) followed by the decode step that
continues all 16 heads by one token from the prefill's final state.
`value` is prefill tokens/s over all ranks (inputs resident in HBM); the
decode workload (256 sequences x 32 heads, 64 chained steps) is reported
alongside as state GB/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own copy of the workload on its own GPU
(independent problems, no data-path collective: weak scaling); a barrier and a
max-over-ranks of the elapsed time bracket the timed region.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from synthetic import decode_inputs, initial_state, prefill_inputs, workload  # noqa: E402

NAMES = ("q", "k", "v", "log_alpha", "beta")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; barrier + max-over-ranks only)
# ----------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 200):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "kda_gated_delta_chunked_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, files):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash(files)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == want:
                return {"bytes_per_launch": float(parts[2]), "scaled_from": " ".join(parts[3:])}
    return None


def make_events(n):
    """Timing events, created eagerly (torch creates the CUDA event on first record)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    return evs


# Algorithmic work per token*head at chunk C, head size d (prefill), and the
# irreducible HBM bytes: q, k, log_alpha (d each) and v (d) and beta read once,
# out written once, all in the input dtype.
def prefill_units(C=64, d=128, esz=2):
    intra_flops = C * (3 * d + 2 * d)             # triangular halves of A, P, T K~, T V, P U
    chain_flops = 6 * d * d                        # W S, Q~ S, K^end^T U
    in_bytes = (4 * d + 1) * esz                   # q, k, log_alpha, v, beta
    out_bytes = d * esz
    return intra_flops, chain_flops, in_bytes, out_bytes


def dense_issued_flops(C=64, d=128):
    """Contraction FLOPs per token and head as the dense products are issued:
    the C x C blocks A and P in full (2 C d each), T K~, T V and P U in full
    (2 C d each), and the three d x d products of the chain (6 d^2)."""
    return 2 * C * d * 2 + 2 * C * d * 3 + 6 * d * d


def bench_workload(args):
    """The prefill workload of the step; ``--tokens T`` keeps its distributions
    and heads but makes it one sequence of T tokens (a smaller profiling case)."""
    w = workload(args.workload)
    if args.tokens:
        w = dataclasses.replace(w, seqlens=[int(args.tokens)], name=f"{w.name}@T{int(args.tokens)}")
    return w


def prefill_launches(N, H, T, C=64, plan_sms=152, min_seg=8):
    """Kernels one bf16 d=128 prefill launches: the sequence table, the
    intra-chunk kernel, the first chain launch, and -- when a sequence is long
    enough to be cut into segments -- the state scan (three or more segments)
    and the output passes of the later segments.  Mirrors the library's plan:
    (N * H) x (segments - 1) CTAs near the SM count, segment 0 about 1.3x the
    others, at least 8 chunks each."""
    chunks = -(-T // C)
    target = plan_sms // max(1, N * H)
    if target < 2 or chunks <= 2 * min_seg:
        return 3
    seg = max(min_seg, (10 * chunks + 10 * target + 12) // (10 * target + 13))
    seg0 = max((13 * seg + 9) // 10, chunks - target * seg)
    segs = 1 if chunks <= seg0 else 1 + -(-(chunks - seg0) // seg)
    return 3 + (1 if segs > 2 else 0) + (1 if segs > 1 else 0)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, dist: Dist):
    import kda_gated_delta_chunked_gb300 as kda

    dev = torch.device("cuda", dist.local if dist.world > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    w = bench_workload(args)
    T, H, D = w.total_tokens, w.num_heads, w.d_k

    files = kda.prefill_kernel_files(w.dtype, D)
    # --- inputs resident in HBM (generated on the device by the seeded generator)
    x = prefill_inputs(w, device=dev)
    s0 = x["initial_state"]
    out = torch.empty((T, H, D), dtype=w.torch_dtype, device=dev)
    sf = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
    desc = kda.make_desc(1, H, D, D, T, w.torch_dtype)
    ws = torch.empty(kda.kda_prefill_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    desc = kda.make_desc(1, H, D, D, T, w.torch_dtype, ws)
    hand = decode_inputs(w if w.decode_seqs else workload(3), 0, device=dev)
    hand = {n: hand[n][:1, :H].contiguous() for n in NAMES}       # one token for each of the H heads
    hand_out = torch.empty((1, H, D), dtype=w.torch_dtype, device=dev)
    ddesc = kda.make_desc(1, H, D, D, 1, w.torch_dtype)
    import ctypes
    ev_store = []

    def step(phase=None):
        if phase is not None:
            arr = (ctypes.c_void_p * 3)(*[e.cuda_event for e in phase])
            ev_store.append(arr)
            desc.phase_events = ctypes.cast(arr, ctypes.c_void_p)
        else:
            desc.phase_events = None
        rc = kda.kda_prefill(desc, x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, s0, out, sf,
                             stream)
        if rc:
            raise kda.KdaError("kda_prefill", rc)
        rc = kda.kda_decode_step(ddesc, *(hand[n] for n in NAMES), sf, hand_out, stream)
        if rc:
            raise kda.KdaError("kda_decode_step", rc)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kda.kda_get_device_status(desc, stream) != kda.KDA_OK:
        raise RuntimeError("device status not OK after warm-up")

    phases = [make_events(3) for _ in range(args.steps)]
    t0, t1 = make_events(2)
    clock = ClockSampler(dev.index, interval_ms=25)     # ~150 ms timed: several samples
    dist.barrier()
    torch.cuda.synchronize()
    clock.start()
    t0.record(stream)
    for i in range(args.steps):
        step(phases[i])
    t1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clocks = clock.stop()
    ms = t0.elapsed_time(t1)
    ms_max = dist.max(ms)
    ms_step = ms_max / args.steps
    intra_ms = statistics.mean(p[0].elapsed_time(p[1]) for p in phases)
    chain_ms = statistics.mean(p[1].elapsed_time(p[2]) for p in phases)
    if kda.kda_get_device_status(desc, stream) != kda.KDA_OK:
        raise RuntimeError("device status not OK after the timed region")

    intra_f, chain_f, in_b, out_b = prefill_units(64, D, 2 if w.dtype == "bf16" else 4)
    units = T * H
    state_bytes = 2 * H * D * D * 4
    tc_peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    kinfo = {
        "intra": {"kernel": "kda intra-chunk (a)", "ms": intra_ms, "bound": "hbm",
                  "achieved": units * in_b / (intra_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                  "unit": "GB/s", "algorithmic_per_launch": units * in_b,
                  "tflops": units * intra_f / (intra_ms * 1e-3) / 1e12,
                  "files": files["intra"]},
        "chain": {"kernel": "kda inter-chunk (b)", "ms": chain_ms, "bound": "tensor",
                  "achieved": units * chain_f / (chain_ms * 1e-3) / 1e12, "peak": tc_peak,
                  "unit": "TFLOP/s", "algorithmic_per_launch": units * chain_f,
                  "gbs": (units * out_b + state_bytes) / (chain_ms * 1e-3) / 1e9,
                  "files": files["chain"]},
    }
    dom = max(kinfo, key=lambda k: kinfo[k]["ms"])
    kd = kinfo[dom]
    tr = measured_traffic(dom, kd["files"])
    roofline = {"bound": kd["bound"], "achieved": round(kd["achieved"], 2), "peak": kd["peak"],
                "unit": kd["unit"], "frac": round(kd["achieved"] / kd["peak"], 4),
                "traffic": None if tr is None else tr["bytes_per_launch"],
                "kernel": kd["kernel"], "peak_source": f"{peak_src} ({'sustained' if kd['bound'] == 'tensor' else 'copy'})",
                "algorithmic_per_launch": kd["algorithmic_per_launch"],
                "launch_ms": round(kd["ms"], 4)}

    res = {
        "metric": "KDA prefill tokens/s (% BF16 TC peak); decode-step state GB/s (% HBM peak)",
        "value": round(T * dist.world / (ms_step * 1e-3), 1),
        "unit": "tokens/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": f"{w.name} + decode hand-off step", "T": T, "H": H, "d_k": D, "d_v": D,
                   "chunk": 64, "inputs": "bf16; state and accumulation fp32",
                   "l2": "inputs (%.1f GB per step) larger than L2; no flush" % (units * (in_b + out_b) / 1e9),
                   "parallelism": f"replicas x{dist.world} (independent problems)"},
        "pct_bf16_tc_peak": round(units * (intra_f + chain_f) / (ms_step * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
        # secondary: the dense products as issued, masked halves included (180,224 FLOP per
        # token and head at C = 64, d = 128)
        "pct_bf16_tc_peak_dense_as_issued": round(units * dense_issued_flops(64, D) / (ms_step * 1e-3) / 1e12
                                                  / peaks["bf16_tflops"], 4),
        "pct_hbm_roofline": round(units * (in_b + out_b) / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "roofline": roofline,
        "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items() if kk != "files"}
                    for k, v in kinfo.items()},
        "gpu_launches": (prefill_launches(1, H, T) + 1) * args.steps,
        "clocks": clocks,
    }

    # --- the same prefill with the scalar (Gated DeltaNet) gate
    if not args.no_scalar_gate:
        res["scalar_gate"] = bench_scalar_gate(kda, args, stream, x, s0, out, sf, ws, w, peaks, peak_src)

    # --- the same prefill filling a prefix cache (state snapshots)
    if not args.no_snapshots:
        res["snapshots"] = bench_snapshots(kda, args, dev, stream, x, s0, out, sf, ws, w, peaks, peak_src, ms_step)

    # --- prefill on the smaller workloads (0: fp32 d = 64, 1: 4,096 tokens, 2: varlen)
    if not args.no_configs:
        res["workloads"] = bench_configs(kda, args, dev, stream, peaks, peak_src)

    # --- reverse mode of the prefill (training), on the 4,096-token workload
    if not args.no_backward:
        res["backward"] = bench_backward(kda, args, dev, stream, peaks, peak_src)

    # --- decode workload (state GB/s)
    if not args.no_decode:
        res["decode"] = bench_decode(kda, args, dev, stream, peaks, peak_src)

    # --- end to end through the C ABI from pinned host buffers
    if not args.no_e2e:
        res["e2e"] = bench_e2e(kda, args, dev, stream, x, s0, w, desc, hand, ddesc)
    del x, out, ws
    torch.cuda.empty_cache()

    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return res


def timed_prefill(kda, desc, args_, stream, steps, warmup):
    """Runs kda_prefill(desc, *args_) warmup + steps times; returns (ms per step,
    mean intra-chunk kernel ms, mean chain ms) from CUDA events on `stream`
    (the library records the phase events between its launches)."""
    import ctypes

    def run(phase=None):
        if phase is not None:
            arr = (ctypes.c_void_p * 3)(*[e.cuda_event for e in phase])
            keep.append(arr)
            desc.phase_events = ctypes.cast(arr, ctypes.c_void_p)
        else:
            desc.phase_events = None
        rc = kda.kda_prefill(desc, *args_, stream) if len(args_) == 9 else \
            kda.kda_prefill_snapshots(desc, *args_, stream)
        if rc:
            raise kda.KdaError("kda_prefill", rc)

    keep = []
    for _ in range(warmup):
        run()
    phases = [make_events(3) for _ in range(steps)]
    t0, t1 = make_events(2)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(steps):
        run(phases[i])
    t1.record(stream)
    torch.cuda.synchronize()
    desc.phase_events = None
    if kda.kda_get_device_status(desc, stream) != kda.KDA_OK:
        raise RuntimeError("device status not OK")
    return (t0.elapsed_time(t1) / steps, statistics.mean(p[0].elapsed_time(p[1]) for p in phases),
            statistics.mean(p[1].elapsed_time(p[2]) for p in phases))


def hbm_roofline(kernel, nbytes, ms, peaks, peak_src):
    a = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(a, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(a / peaks["hbm_gbs"], 4), "traffic": None, "kernel": kernel,
            "peak_source": f"{peak_src} (copy)", "algorithmic_per_launch": nbytes, "launch_ms": round(ms, 4)}


def bench_scalar_gate(kda, args, stream, x, s0, out, sf, ws, w, peaks, peak_src):
    """Prefill tokens/s of the same inputs with one gate per (token, head)
    (channel 0 of log_alpha), the Gated DeltaNet form; kernel (a) against HBM
    on its algorithmic bytes (q, k, v per channel, one log alpha and one beta
    per token and head)."""
    T, H, D = w.total_tokens, w.num_heads, w.d_k
    la = x["log_alpha"][:, :, 0].contiguous()
    desc = kda.make_desc(1, H, D, D, T, w.torch_dtype, ws, flags=kda.KDA_FLAG_SCALAR_GATE)
    steps = max(3, min(args.steps, 5))
    ms, intra_ms, chain_ms = timed_prefill(kda, desc, (x["q"], x["k"], x["v"], la, x["beta"], None, s0, out, sf),
                                           stream, steps, args.warmup)
    del la
    esz = 2 if w.dtype == "bf16" else 4
    per_tok = (3 * D + 2) * esz                     # q, k, v rows; one log alpha and one beta
    return {"workload": f"{w.name}, log_alpha one per (token, head)", "value": round(T / (ms * 1e-3), 1),
            "unit": "tokens/s", "ms_per_step": round(ms, 4), "steps": steps,
            "intra_ms": round(intra_ms, 4), "chain_ms": round(chain_ms, 4),
            "roofline": hbm_roofline("kda intra-chunk (a), scalar gate", T * H * per_tok, intra_ms, peaks, peak_src),
            "gpu_launches": prefill_launches(1, H, T) * steps}


def bench_snapshots(kda, args, dev, stream, x, s0, out, sf, ws, w, peaks, peak_src, plain_ms, every=4096):
    """The same prefill saving the state after every `every` tokens (a prefix
    cache filled during the prefill): step time against the plain prefill and
    kernel (a) against HBM as in the main line."""
    T, H, D = w.total_tokens, w.num_heads, w.d_k
    at = torch.tensor([[0, p] for p in range(every, T + 1, every)], dtype=torch.int32, device=dev)
    m = at.shape[0]
    snaps = torch.empty((m, H, D, D), dtype=torch.float32, device=dev)
    desc = kda.make_desc(1, H, D, D, T, w.torch_dtype, ws)
    steps = max(3, min(args.steps, 5))
    ms, intra_ms, chain_ms = timed_prefill(
        kda, desc, (x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, s0, out, sf, m, at, snaps),
        stream, steps, args.warmup)
    in_b = prefill_units(64, D, 2 if w.dtype == "bf16" else 4)[2]
    res = {"workload": f"{w.name}, state saved every {every} tokens ({m} snapshots, "
                       f"{m * H * D * D * 4 / 1e9:.2f} GB)",
           "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "overhead_vs_plain": round(ms / plain_ms - 1.0, 4), "steps": steps,
           "intra_ms": round(intra_ms, 4), "chain_ms": round(chain_ms, 4),
           "roofline": hbm_roofline("kda intra-chunk (a)", T * H * in_b, intra_ms, peaks, peak_src),
           "gpu_launches": (prefill_launches(1, H, T) + 1) * steps}
    del snaps, at
    return res


def fp32_alu_peak(peaks):
    """fp32 FMA peak of the CUDA cores: SMs x 128 fp32 lanes x 2 FLOP x max SM clock."""
    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    mhz = peaks.get("sm_max_mhz", 2070.0)
    return p.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12


# Contractions of the chunked reverse mode per token*head (chunk C, head size
# d), counted as the tensor cores issue them on the rows that carry results:
# the forward recomputation (its dense-as-issued count, 180,224 at C=64,
# d=128), the reverse chain over chunks (K^end dS' and [W; Q']^T [-K^end dS';
# dO]: 6 d^2) and the per-chunk gradient products: G and Q~K^^T (4 C d),
# T [K~ | V] (4 C d), W S (2 d^2), K^end dS' + P^T dO (2 d^2 + 2 C d),
# U dS'^T (2 d^2), [dO; dU] S^T (4 d^2), dO U^T (2 C d), dW K~^T + dU V^T
# (4 C d), T^T dU and T^T dW (4 C d), [dP; dG] K^ (4 C d), dP^T Q~ + dG^T K~
# (4 C d).  The fp32 64 x 64 products behind dA and the solve are not counted.
def backward_tc_flop_per_token(C=64, d=128):
    fwd = dense_issued_flops(C, d)
    chain = 6 * d * d
    chunk = 28 * C * d + 10 * d * d
    return fwd + chain + chunk


def bench_backward(kda, args, dev, stream, peaks, peak_src):
    """Prefill reverse mode on workload 1: tokens/s of the tensor-core backward
    (forward recomputation saving every chunk's state, the reverse chain, the
    per-chunk gradient kernel) against the burst bf16 peak on its contraction
    FLOPs, with the fp32 CUDA-core backward timed beside it."""
    w = workload(1)
    T, H, D = w.total_tokens, w.num_heads, w.d_k
    x = prefill_inputs(w, device=dev)
    gen = torch.Generator(device=dev).manual_seed(7)
    do = torch.randn((T, H, D), generator=gen, device=dev, dtype=torch.float32).to(w.torch_dtype)
    dfin = torch.randn((1, H, D, D), generator=gen, device=dev, dtype=torch.float32)
    f32 = dict(dtype=torch.float32, device=dev)
    g = [torch.empty((T, H, D), **f32) for _ in range(4)] + [torch.empty((T, H), **f32),
                                                             torch.empty((1, H, D, D), **f32)]

    def timed(flags):
        desc = kda.make_desc(1, H, D, D, T, w.torch_dtype, flags=flags)
        ws = torch.empty(kda.kda_backward_workspace_bytes(desc), dtype=torch.uint8, device=dev)
        desc = kda.make_desc(1, H, D, D, T, w.torch_dtype, ws, flags=flags)

        def run():
            rc = kda.kda_prefill_backward(desc, x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None,
                                          x["initial_state"], do, dfin, *g, stream)
            if rc:
                raise kda.KdaError("kda_prefill_backward", rc)

        for _ in range(max(2, args.warmup)):
            run()
        steps = 5
        t0, t1 = make_events(2)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(steps):
            run()
        t1.record(stream)
        torch.cuda.synchronize()
        if kda.kda_get_device_status(desc, stream) != kda.KDA_OK:
            raise RuntimeError("device status not OK (backward)")
        del ws
        return t0.elapsed_time(t1) / steps, steps

    ms, steps = timed(0)
    ms_cc, _ = timed(kda.KDA_FLAG_CUDA_CORE_PREFILL)
    per_tok = backward_tc_flop_per_token(64, D)
    flop = per_tok * T * H
    peak = peaks["bf16_tflops"]
    ach = flop / (ms * 1e-3) / 1e12
    # sequence table, slot table, forward (intra + chain launches), reverse chain,
    # per-chunk kernel, and the CUDA-core fallback's two launches (which return at once)
    launches = 2 + (prefill_launches(1, H, T) - 1) + 2 + 2
    return {"workload": w.name, "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 4), "steps": steps, "gpu_launches": launches * steps,
            "path": "tensor cores (bf16 operands, fp32 accumulation)",
            "roofline": {"bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(ach / peak, 4), "traffic": None,
                         "kernel": "kda backward, whole call (forward recompute + reverse chain + per-chunk gradients)",
                         "peak_source": f"{peak_src} (bf16 burst)", "algorithmic_per_launch": flop,
                         "flop_per_token_head": per_tok, "launch_ms": round(ms, 4)},
            "cuda_core": {"ms_per_step": round(ms_cc, 4), "value": round(T / (ms_cc * 1e-3), 1),
                          "unit": "tokens/s", "speedup_of_tensor_cores": round(ms_cc / ms, 2)},
            "note": "gradients of q, k, v, log_alpha, beta and the initial state"}


def bench_configs(kda, args, dev, stream, peaks, peak_src, indices=(0, 1, 2)):
    """Prefill throughput on the smaller workloads (0: one fp32 sequence, d = 64,
    on the CUDA-core path; 1: 4,096 tokens x 16 heads; 2: the 8-sequence varlen
    batch x 32 heads): tokens/s per call, the two kernels' times, and kernel (a)
    against HBM on its input bytes.  Their inputs fit in L2, so a buffer twice
    its size is written before every timed call (outside the call's events)."""
    import ctypes
    res = {}
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size, dtype=torch.uint8, device=dev)
    steps = 10
    for idx in indices:
        w = workload(idx)
        T, H, D, Dv, N = w.total_tokens, w.num_heads, w.d_k, w.d_v, w.num_seqs
        x = prefill_inputs(w, device=dev)
        o = torch.empty((T, H, Dv), dtype=w.torch_dtype, device=dev)
        sf = torch.empty((N, H, D, Dv), dtype=torch.float32, device=dev)
        desc = kda.make_desc(N, H, D, Dv, T, w.torch_dtype)
        ws = torch.empty(kda.kda_prefill_workspace_bytes(desc), dtype=torch.uint8, device=dev)
        desc = kda.make_desc(N, H, D, Dv, T, w.torch_dtype, ws)
        call = (x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"], x["initial_state"], o, sf)
        for _ in range(3):
            rc = kda.kda_prefill(desc, *call, stream)
            if rc:
                raise kda.KdaError("kda_prefill", rc)
        ev = [make_events(5) for _ in range(steps)]
        keep = []
        torch.cuda.synchronize()
        for e in ev:
            flush.zero_()
            arr = (ctypes.c_void_p * 3)(*[x_.cuda_event for x_ in e[1:4]])
            keep.append(arr)
            desc.phase_events = ctypes.cast(arr, ctypes.c_void_p)
            e[0].record(stream)
            rc = kda.kda_prefill(desc, *call, stream)
            e[4].record(stream)
            if rc:
                raise kda.KdaError("kda_prefill", rc)
        torch.cuda.synchronize()
        desc.phase_events = None
        if kda.kda_get_device_status(desc, stream) != kda.KDA_OK:
            raise RuntimeError(f"device status not OK (workload {idx})")
        ms = statistics.mean(e[0].elapsed_time(e[4]) for e in ev)
        intra = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
        chain = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
        esz = 2 if w.dtype == "bf16" else 4
        in_b = (4 * D + 1) * esz if Dv == D else (3 * D + Dv + 1) * esz
        tc = w.dtype == "bf16" and D == 128
        res[str(idx)] = {"workload": w.name, "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s",
                         "ms_per_call": round(ms, 4), "intra_ms": round(intra, 4), "chain_ms": round(chain, 4),
                         "path": "tensor cores" if tc else "CUDA cores (fp32)", "steps": steps,
                         "roofline": hbm_roofline("kda intra-chunk (a)" + ("" if tc else ", CUDA cores"),
                                                  T * H * in_b, intra, peaks, peak_src),
                         "l2": "flushed before each call"}
        del x, o, sf, ws
    del flush
    torch.cuda.empty_cache()
    return res


def bench_decode(kda, args, dev, stream, peaks, peak_src):
    w = workload(3)
    N, H, D = w.decode_seqs, w.num_heads, w.d_k
    state = initial_state(w, N, device=dev)
    steps = [decode_inputs(w, s, device=dev) for s in range(w.decode_steps)]
    outs = torch.empty((w.decode_steps, N, H, D), dtype=w.torch_dtype, device=dev)
    desc = kda.make_desc(N, H, D, D, N, w.torch_dtype)

    def run():
        for s in range(w.decode_steps):
            x = steps[s]
            rc = kda.kda_decode_step(desc, *(x[n] for n in NAMES), state, outs[s], stream)
            if rc:
                raise kda.KdaError("kda_decode_step", rc)

    for _ in range(max(1, args.warmup)):
        run()
    torch.cuda.synchronize()
    reps = max(1, args.decode_reps)
    t0, t1 = make_events(2)
    clock = ClockSampler(dev.index, interval_ms=50)      # the region is ~0.5 s: several samples
    clock.start()
    t0.record(stream)
    for _ in range(reps):
        run()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = clock.stop()
    ms = t0.elapsed_time(t1) / (reps * w.decode_steps)
    state_bytes = 2 * N * H * D * D * 4
    io_bytes = N * H * (4 * D + 1) * 2 + N * H * D * 2
    gbs = state_bytes / (ms * 1e-3) / 1e9
    return {"workload": w.name, "metric": "decode-step state GB/s", "value": round(gbs, 1), "unit": "GB/s",
            "steps_per_s": round(1e3 / ms, 1), "us_per_step": round(ms * 1e3, 2),
            "total_gbs_incl_io": round((state_bytes + io_bytes) / (ms * 1e-3) / 1e9, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": None,
                         "peak_source": peak_src, "algorithmic_per_launch": state_bytes},
            "l2": "state (%.2f GB) larger than L2; no flush" % (state_bytes / 2e9),
            "gpu_launches": reps * w.decode_steps, "clocks": clocks}


def bench_e2e(kda, args, dev, stream, x, s0, w, desc, hand, ddesc):
    """Same metric through the public C ABI with pinned HOST buffers.  Every
    step copies all inputs host->device, runs the prefill plus the decode
    hand-off, and reads the outputs and final state back device->host.  The
    sequence is processed in `pieces` consecutive calls, each continuing from
    the previous call's final state in place (the state hand-off the API
    exposes), so that the copies of one piece overlap the compute of the next
    on separate streams."""
    T, H, D = w.total_tokens, w.num_heads, w.d_k
    pieces = max(1, args.e2e_pieces)
    while T % (pieces * 64):
        pieces -= 1
    tp = T // pieces
    hx = {n: torch.empty(x[n].shape, dtype=x[n].dtype, pin_memory=True) for n in NAMES}
    for n in NAMES:
        hx[n].copy_(x[n])
    hs0 = torch.empty(s0.shape, dtype=s0.dtype, pin_memory=True)
    hs0.copy_(s0)
    hout = torch.empty((T, H, D), dtype=w.torch_dtype).pin_memory()
    hsf = torch.empty((1, H, D, D), dtype=torch.float32).pin_memory()
    hho = torch.empty((1, H, D), dtype=w.torch_dtype).pin_memory()
    dx = {n: torch.empty_like(x[n]) for n in NAMES}
    dst = torch.empty_like(s0)
    dout = torch.empty((T, H, D), dtype=w.torch_dtype, device=dev)
    dho = torch.empty((1, H, D), dtype=w.torch_dtype, device=dev)
    pdesc = kda.make_desc(1, H, D, D, tp, w.torch_dtype)
    pws = torch.empty(kda.kda_prefill_workspace_bytes(pdesc), dtype=torch.uint8, device=dev)
    pdesc = kda.make_desc(1, H, D, D, tp, w.torch_dtype, pws)
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d = sum(hx[n].numel() * hx[n].element_size() for n in NAMES) + hs0.numel() * 4
    d2h = hout.numel() * hout.element_size() + hsf.numel() * 4 + hho.numel() * hho.element_size()

    spans = []                             # (first H2D start, last H2D end) events per step
    # events for those spans, created (and synchronised) before anything is timed
    span_pool = iter([make_events(2) for _ in range(2 + max(1, args.e2e_steps))])

    def step():
        h2d_s.wait_stream(stream)          # the previous step no longer reads the device inputs
        e_h0, e_h1 = next(span_pool)
        with torch.cuda.stream(h2d_s):
            e_h0.record(h2d_s)
            dst.copy_(hs0, non_blocking=True)
        ev_in, ev_out = [], []
        for k in range(pieces):
            a, b = k * tp, (k + 1) * tp
            with torch.cuda.stream(h2d_s):
                for n in NAMES:
                    dx[n][a:b].copy_(hx[n][a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d_s)
                ev_in.append(e)
        e_h1.record(h2d_s)
        spans.append((e_h0, e_h1))
        for k in range(pieces):
            a, b = k * tp, (k + 1) * tp
            stream.wait_event(ev_in[k])
            rc = kda.kda_prefill(pdesc, dx["q"][a:b], dx["k"][a:b], dx["v"][a:b], dx["log_alpha"][a:b],
                                 dx["beta"][a:b], None, dst, dout[a:b], dst, stream)
            if rc:
                raise kda.KdaError("kda_prefill", rc)
            e = torch.cuda.Event()
            e.record(stream)
            ev_out.append(e)
        rc = kda.kda_decode_step(ddesc, *(hand[n] for n in NAMES), dst, dho, stream)
        if rc:
            raise kda.KdaError("kda_decode_step", rc)
        done = torch.cuda.Event()
        done.record(stream)
        with torch.cuda.stream(d2h_s):
            for k in range(pieces):
                a, b = k * tp, (k + 1) * tp
                d2h_s.wait_event(ev_out[k])
                hout[a:b].copy_(dout[a:b], non_blocking=True)
            d2h_s.wait_event(done)
            hsf.copy_(dst, non_blocking=True)
            hho.copy_(dho, non_blocking=True)
        stream.wait_stream(d2h_s)

    for _ in range(2):                     # warm-up: first DMA over freshly pinned pages
        step()
    torch.cuda.synchronize()
    # The host link's own rate right now (1 GiB of q's own bytes copied each
    # way, values unchanged), so a run on a box whose host side is busy can be
    # told from a slow pipeline.
    probe = hx["q"].view(-1)[: min(hx["q"].numel(), 1 << 29)]
    dprobe = dx["q"].view(-1)[: probe.numel()]
    link = {}
    for name, (dst_t, src_t) in (("h2d_gbs", (dprobe, probe)), ("d2h_gbs", (probe, dprobe))):
        a, b = make_events(2)
        a.record(stream)
        dst_t.copy_(src_t, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        link[name] = round(probe.numel() * probe.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    # Both directions at once, as the pipeline runs them (H2D of q into dx["q"],
    # D2H of dx["k"] into hx["k"]: each buffer receives its own bytes back).
    pk = hx["k"].view(-1)[: probe.numel()]
    dk = dx["k"].view(-1)[: probe.numel()]
    a, b = make_events(2)
    torch.cuda.synchronize()
    a.record(stream)
    h2d_s.wait_stream(stream)
    d2h_s.wait_stream(stream)
    with torch.cuda.stream(h2d_s):
        dprobe.copy_(probe, non_blocking=True)
    with torch.cuda.stream(d2h_s):
        pk.copy_(dk, non_blocking=True)
    stream.wait_stream(h2d_s)
    stream.wait_stream(d2h_s)
    b.record(stream)
    torch.cuda.synchronize()
    link["both_ways_gbs"] = round(2 * probe.numel() * probe.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    # Each input copied whole (host to device), to show whether some of the
    # pinned host memory is slower than the 1 GiB probed above.
    per = {}
    for n in NAMES:
        a, b = make_events(2)
        a.record(stream)
        dx[n].copy_(hx[n], non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        per[n] = round(hx[n].numel() * hx[n].element_size() / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    link["h2d_gbs_whole_inputs"] = per
    steps = max(1, args.e2e_steps)
    t0, t1 = make_events(2)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - w0) / steps
    ms = t0.elapsed_time(t1) / steps
    h2d_ms = statistics.mean(a.elapsed_time(b) for a, b in spans[-steps:])
    link["h2d_gbs_in_timed_steps"] = round(h2d / (h2d_ms * 1e-3) / 1e9, 1)
    return {"value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3), "wall_ms_per_step": round(wall * 1e3, 3),
            "steps": steps, "host_buffers": "pinned", "link_probe": link,
            "pieces": pieces, "schedule": "H2D, prefill continuation and D2H of consecutive pieces overlap "
                                          "on three streams"}


def cpu_baseline(w, seconds):
    """The fp64 oracle, as it stands, on the host cores: a bounded sample of the
    workload (its first tokens, all heads)."""
    import oracle
    x = None
    n_tok = 256
    spent = 0.0
    # grow the sample until one run takes a meaningful time, then take the one
    # whose estimated cost is about `seconds`
    while True:
        x = prefill_inputs(w, t_range=(0, n_tok))
        s0 = x["initial_state"]
        t = time.perf_counter()
        oracle.prefill(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, s0)
        spent = time.perf_counter() - t
        if spent >= seconds / 4 or n_tok >= w.total_tokens:
            break
        n_tok = min(w.total_tokens, n_tok * 4)
    if spent < seconds / 2 and n_tok < w.total_tokens:
        n_tok = min(w.total_tokens, int(n_tok * seconds / max(spent, 1e-3)))
        x = prefill_inputs(w, t_range=(0, n_tok))
        t = time.perf_counter()
        oracle.prefill(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, x["initial_state"])
        spent = time.perf_counter() - t
    # the same oracle on one core, on a sample a sixteenth as long
    n1 = max(64, n_tok // 16)
    x1 = prefill_inputs(w, t_range=(0, n1))
    t = time.perf_counter()
    oracle.prefill(x1["q"], x1["k"], x1["v"], x1["log_alpha"], x1["beta"], None, x1["initial_state"], threads=1)
    spent1 = time.perf_counter() - t
    return {"value": round(n_tok / spent, 2), "unit": "tokens/s", "cores": oracle.default_threads(),
            "kind": "oracle", "seconds": round(spent, 2),
            "sample": f"first {n_tok} tokens x {w.num_heads} heads of {w.name} (fp64 recurrence, "
                      f"threads over head x column block)",
            "one_core": {"value": round(n1 / spent1, 2), "unit": "tokens/s", "cores": 1,
                         "sample": f"first {n1} tokens x {w.num_heads} heads", "seconds": round(spent1, 2)}}


# ----------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ----------------------------------------------------------------------------
def run_reference(args):
    import oracle
    w = bench_workload(args)
    n_tok = args.ref_tokens
    chunks = [prefill_inputs(w, t_range=(i * n_tok, (i + 1) * n_tok)) for i in range(2)]
    s0 = chunks[0]["initial_state"]

    def step(i):
        x = chunks[i % 2]
        oracle.prefill(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None, s0)

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t
    value = n_tok * args.steps / el
    return {
        "impl": "reference",
        "metric": "KDA prefill tokens/s (% BF16 TC peak); decode-step state GB/s (% HBM peak)",
        "value": round(value, 2), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": f"{w.name} + decode hand-off step", "T": w.total_tokens, "H": w.num_heads,
                   "d_k": w.d_k, "d_v": w.d_v, "chunk": 64},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": oracle.default_threads(),
                         "kind": "oracle",
                         "sample": f"each step: {n_tok} tokens x {w.num_heads} heads of {w.name}"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4)
    ap.add_argument("--tokens", type=int, default=0,
                    help="one sequence of this many tokens with the workload's distributions (profiling case)")
    ap.add_argument("--decode-reps", type=int, default=48)   # 48 x 64 steps, ~0.5 s timed
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-pieces", type=int, default=16)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=2048)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-scalar-gate", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-snapshots", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the prefill's reverse mode (workload 1) and print its JSON object")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return
    if args.backward_only:
        import kda_gated_delta_chunked_gb300 as kda
        torch.cuda.set_device(0)
        peaks, peak_src = load_peaks()
        print(json.dumps(bench_backward(kda, args, torch.device("cuda", 0), torch.cuda.current_stream(), peaks,
                                        peak_src)))
        return
    dist = Dist()
    try:
        res = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(res))
    finally:
        dist.close()


if __name__ == "__main__":
    main()
