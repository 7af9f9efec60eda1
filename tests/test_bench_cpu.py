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


def test_traffic_files_are_consistent():
    """Every committed DRAM-traffic summary names its workload and variant as
    its file does, its algorithmic bytes are the workload's (inputs and
    outputs of a full launch), its total is read + write, its command runs
    committed files only, and bench.py uses it exactly when it was taken on
    the current kernel sources."""
    import glob
    import os
    import re
    files = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "fused_mlp_*.traffic.json")))
    assert len(files) >= 5
    for path in files:
        d = json.load(open(path))
        m = re.fullmatch(r"fused_mlp_([a-z0-9]+)_([a-z_]+)\.traffic\.json", os.path.basename(path))
        assert m and (d["variant"], d["workload"]) == (m.group(1), m.group(2)), path
        w = synth.WORKLOADS[d["workload"]]
        assert d["algorithmic_bytes_per_launch"] == w.n_evals * w.hbm_bytes_per_eval, path
        assert d["dram_bytes_per_launch"] == pytest.approx(
            d["dram_bytes_read_per_launch"] + d["dram_bytes_write_per_launch"], abs=2), path
        assert re.fullmatch(r"[0-9a-f]{64}", d["kernel_sources_sha256"])
        assert "--clock-control none" in d["command"] and "python bench.py" in d["command"]
        assert "_work" not in d["command"]
        current = d["kernel_sources_sha256"] == bench.kernel_sources_sha()
        got = bench.load_traffic(d["workload"], d["variant"])
        assert got == (d["dram_bytes_per_launch"] if current else None), path
