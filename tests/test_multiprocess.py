"""The multi-rank plumbing of bench.py on CPU: two gloo ranks (127.0.0.1).
The path shards into independent problems, so ranks only meet at a barrier
and a max over their elapsed times; the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import sys, time
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
d.barrier()
r = d.rank
m = d.max(1.5 * (r + 1))
d.barrier()
print("RESULT", d.rank, d.world, m, flush=True)
d.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    env = dict(os.environ)
    env.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "CUDA_VISIBLE_DEVICES": ""})
    return env


def test_two_gloo_ranks_barrier_and_max():
    port = _free_port()
    code = RANK_SCRIPT.format(root=ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code], env=_env(r, 2, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    results = sorted(line.split()[1:] for out, _ in outs for line in out.splitlines() if line.startswith("RESULT"))
    assert results == [["0", "2", "3.0"], ["1", "2", "3.0"]]   # every rank sees the max over ranks


def test_reference_arm_runs_on_rank0_only():
    port = _free_port()
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
            "--steps", "1", "--warmup", "3", "--ref-tokens", "64"]
    procs = [subprocess.Popen(args, env=_env(r, 2, port), stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True, cwd=ROOT) for r in range(2)]
    outs = [p.communicate(timeout=300) for p in procs]
    assert all(p.returncode == 0 for p in procs), [e for _, e in outs]
    line0 = [l for l in outs[0][0].splitlines() if l.startswith("{")]
    assert len(line0) == 1 and outs[1][0].strip() == ""
    rec = json.loads(line0[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["e2e"]["h2d_bytes_per_step"] == 0
