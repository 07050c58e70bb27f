"""Write tests/golden/tiny_frames.json from the CPU oracle alone.

The tiny Dual-AR model (2+2 layers, hidden 256), seed 0: prefill 16 prompt
ids, then 8 decode frames, greedy and top-k 30 (Philox seed 1234).  Run from
the repository root:  python tests/golden/make_tiny_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from synth import TINY, make_weights, make_prompt  # noqa: E402


def run(sampling):
    o = oracle.DualAROracle(TINY, make_weights(TINY, 0))
    f, z = o.prefill(make_prompt(TINY, 16, seed=0), sampling)
    frames, sums = [f[0].tolist()], [float(np.sum(z))]
    for _ in range(8):
        f, z = o.decode_frame(sampling)
        frames.append(f[0].tolist())
        sums.append(float(np.sum(z)))
    return frames, sums


def main():
    g_frames, g_sums = run(None)
    k_frames, _ = run({"top_k": 30, "seed": 1234})
    out = {
        "source": "written by tests/golden/make_tiny_golden.py from the CPU oracle",
        "workload": "tiny bf16 2+2 layers, hidden 256, seed 0, prefill 16 + decode 8",
        "greedy_frames": g_frames,
        "greedy_logit_sums": g_sums,
        "topk30_seed1234_frames": k_frames,
    }
    with open(os.path.join(HERE, "tiny_frames.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
