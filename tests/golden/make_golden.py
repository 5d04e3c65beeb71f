"""Writes tests/golden/tiny_seed0.json from the CPU oracle only.

The fixture locks the oracle's output on the tiny layer shape (H=256, E=8,
k=2, I=128, m=16, seed 0) so that an accidental change to the oracle's
arithmetic shows up as a failing test.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mixture_experts_ffn_gemv_gb300 import inputs as I  # noqa: E402


def main():
    wl = I.WORKLOADS["tiny"]
    layer = I.make_layer(wl, seed=0)
    x = I.make_x(wl.shape, 16, seed=0)
    r = oracle.reference(wl.shape, layer, x)
    rows = [0, 5, 15]
    doc = {
        "what": "oracle output on the tiny MoE layer (H=256, E=8, top_k=2, I=128, m=16, seed 0)",
        "written_by": "tests/golden/make_golden.py (calls only oracle/)",
        "x_digest": hashlib.sha256(x.view(torch.int16).numpy().tobytes()).hexdigest()[:16],
        "ids": r["ids"].tolist(),
        "w": [[float(v) for v in row] for row in r["w"]],
        "rows": rows,
        "out_rows": [[float(v) for v in r["out"][t]] for t in rows],
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_seed0.json"), "w") as f:
        json.dump(doc, f, indent=0)


if __name__ == "__main__":
    main()
