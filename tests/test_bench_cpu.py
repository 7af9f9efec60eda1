"""bench.py on the CPU: the reference arm's JSON line and the roofline terms
the GPU arm reports (no GPU needed)."""
import json

import pytest

import bench
from mlp_neural_gb300 import synth


def test_reference_arm_line(capsys):
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1",
                       "--warmup", "0"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 0
    assert line["value"] > 0
    assert line["config"]["workload"] == "tiny"
    assert line["config"]["dims"] == list(synth.WORKLOADS["tiny"].dims)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_cores() and cb["value"] == line["value"]
    assert "threads" in cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("name,bound", [("tiny", "hbm"), ("page", "tensor"),
                                        ("ablation", "tensor"), ("wide", "tensor"),
                                        ("hetero", "tensor")])
def test_roofline_bound_per_workload(name, bound):
    # Arithmetic intensity (FLOPs per HBM byte) against the ridge point of
    # the fallback peaks: 160 for the tiny network is below it, the others
    # (448, 1,357, 2,112) are above.
    w = synth.WORKLOADS[name]
    got, t_tensor, t_hbm = bench.roofline_bound(w, dict(bench.FALLBACK_PEAKS))
    assert got == bound
    assert t_tensor == pytest.approx(w.flops_per_eval / (bench.FALLBACK_PEAKS["bf16_tflops"] * 1e12))
    assert t_hbm == pytest.approx(w.hbm_bytes_per_eval / (bench.FALLBACK_PEAKS["hbm_gbs"] * 1e9))


def test_algorithmic_units_per_evaluation():
    # 2 * sum(K_l * N_l) FLOPs and 2 * (d0 + dL) bytes per evaluation.
    for name, flops, hbm in [("tiny", 15360, 96), ("page", 57344, 128), ("wide", 217088, 160),
                             ("hetero", 337920, 160)]:
        w = synth.WORKLOADS[name]
        assert w.flops_per_eval == flops and w.hbm_bytes_per_eval == hbm
