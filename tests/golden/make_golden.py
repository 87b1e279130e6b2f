"""Write the oracle golden fixtures in this folder.

Calls only the fp64 oracle (and the seeded input generator for its inputs).
Each fixture records sampled entries and norms of the oracle's output and
final state for one seeded workload, so that any later change to the
oracle's arithmetic (or to the generator) shows up as a diff here.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from synthetic import custom, prefill_inputs, workload  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))

CASES = {
    # 256-token, 2-head, d=64 fp32 workload with a zero initial state.
    "oracle_single_T256_H2_d64_f32": lambda: workload(0),
    # ragged varlen bf16 case: several chunks, partial tails, an empty and a 1-token sequence.
    "oracle_varlen_ragged_H3_d128_bf16": lambda: custom(21, [150, 0, 1, 64, 200], 3, 128, "bf16"),
}


def fixture(w):
    d = prefill_inputs(w)
    out, sf = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                             d["cu_seqlens"], d["initial_state"])
    rng = np.random.default_rng(0)
    oi = [tuple(int(rng.integers(0, s)) for s in out.shape) for _ in range(24)] if out.size else []
    si = [tuple(int(rng.integers(0, s)) for s in sf.shape) for _ in range(24)]
    return {
        "workload": w.name, "seed": w.seed, "seqlens": w.seqlens, "num_heads": w.num_heads,
        "d_k": w.d_k, "d_v": w.d_v, "dtype": w.dtype,
        "out_norm": float(np.linalg.norm(out)), "state_norm": float(np.linalg.norm(sf)),
        "out_samples": [[list(i), repr(float(out[i]))] for i in oi],
        "state_samples": [[list(i), repr(float(sf[i]))] for i in si],
    }


if __name__ == "__main__":
    for name, mk in CASES.items():
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(fixture(mk()), f, indent=1)
        print("wrote", name)
