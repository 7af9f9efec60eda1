"""Writes tests/golden/oracle_regression.json from the oracle alone.

Run: python tests/golden/make_golden.py
It calls only oracle/ and the seeded generator; no GPU code is involved. The
file guards the oracle against unintended changes: test_golden.py recomputes
the same rows and compares bit for bit.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mlp_neural_gb300 import synth  # noqa: E402

ROWS = [0, 1, 2, 127, 128, 65535]


def compute():
    out = {}
    for name in ("tiny", "page", "hetero"):
        w = synth.WORKLOADS[name]
        W, b = synth.net_params(w.dims, w.seed)
        rows = {}
        for r in ROWS:
            x = synth.inputs(w, r, 1)
            y = oracle.forward(w.dims, W, b, x)[0]
            rows[str(r)] = [f"{int(v):04x}" for v in y]
        out[name] = {"dims": list(w.dims), "seed": w.seed, "rows": rows}
    return out


def compute_fp8():
    """The E4M3 pass (layers 2..L in E4M3) of the two wide networks, and a
    SHA-256 of their E4M3 weight images."""
    import hashlib
    out = {}
    for name in ("wide", "hetero"):
        w = synth.WORKLOADS[name]
        W, b = synth.net_params(w.dims, w.seed)
        rows = {}
        for r in ROWS:
            x = synth.inputs(w, r, 1)
            y = oracle.forward_fp8(w.dims, W, b, x)[0]
            rows[str(r)] = [f"{int(v):04x}" for v in y]
        images = hashlib.sha256(oracle.pack_fp8(w.dims, W).tobytes()).hexdigest()
        out[name] = {"dims": list(w.dims), "seed": w.seed, "rows": rows, "images_sha256": images}
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump({"generator": "tests/golden/make_golden.py (oracle only)", "workloads": compute(),
                   "fp8_workloads": compute_fp8()}, f, indent=1)
    print("wrote", path)
