"""Golden fixtures: the page's printed constants and the oracle regression file."""
import json
import os

import numpy as np

from mlp_neural_gb300 import synth

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def test_page_workload_counts():
    g = _load("page_constants.json")
    assert g["fixed_inputs"] * g["repeats_per_dispatch"] == g["evals_per_dispatch"]
    w = synth.WORKLOADS["page"]
    assert (w.n_unique, w.repeats, w.n_evals) == (
        g["fixed_inputs"], g["repeats_per_dispatch"], g["evals_per_dispatch"])


def test_page_slope_constant(orc):
    g = _load("page_constants.json")
    assert g["activation_slope_literal"] == "half(0.01)"
    assert orc.slope_f16() == int(np.float16(g["activation_slope_value"]).view(np.uint16))


def test_page_throughput_arithmetic():
    # M eval/s = evaluations / seconds / 1e6, as the page prints them.
    g = _load("page_constants.json")
    for p in g["passes"]:
        meps = g["evals_per_dispatch"] / (p["median_ms"] * 1e-3) / 1e6
        assert round(meps, 2) == p["M_eval_per_s"], p
    t = {p["variant"]: p["median_ms"] for p in g["passes"]}
    bad, good, opt = (t["indexed lanes, row-major weights"], t["native max, row-major weights"],
                      t["native max, InferencingOptimal weights"])
    assert round(bad / good, 3) == g["speedup_native_vs_indexed"]
    assert round(100 * (1 - opt / good), 2) == g["time_reduction_optimal_vs_rowmajor_percent"]


def test_oracle_regression(orc):
    g = _load("oracle_regression.json")["workloads"]
    for name, rec in g.items():
        w = synth.WORKLOADS[name]
        assert list(w.dims) == rec["dims"] and w.seed == rec["seed"]
        W, b = synth.net_params(w.dims, w.seed)
        for r, hexes in rec["rows"].items():
            y = orc.forward(w.dims, W, b, synth.inputs(w, int(r), 1))[0]
            assert [f"{int(v):04x}" for v in y] == hexes, (name, r)


def test_oracle_fp8_regression(orc):
    """The oracle's E4M3 pass and its E4M3 images, against the stored values."""
    import hashlib
    g = _load("oracle_regression.json")["fp8_workloads"]
    assert set(g) == {"wide", "hetero"}
    for name, rec in g.items():
        w = synth.WORKLOADS[name]
        assert list(w.dims) == rec["dims"] and w.seed == rec["seed"]
        W, b = synth.net_params(w.dims, w.seed)
        assert hashlib.sha256(orc.pack_fp8(w.dims, W).tobytes()).hexdigest() == rec["images_sha256"]
        for r, hexes in rec["rows"].items():
            y = orc.forward_fp8(w.dims, W, b, synth.inputs(w, int(r), 1))[0]
            assert [f"{int(v):04x}" for v in y] == hexes, (name, r)
