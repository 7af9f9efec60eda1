"""The checking build (libnmmlp_check.so, kernels compiled with
NM_RANGE_CHECKS) on the GPU.

Its kernels compare every tensor-memory column range and every shared-memory
range they touch with the plan's limits and flag a miss in the status word,
without changing any access. So, run in a child process with NM_CHECKED=1
(one process holds one of the two libraries):
 - every kernel instantiation (resident fused, row-major, scalar-activation,
   paired-tiles; streamed, streamed with A split between TMEM and shared
   memory, streamed scalar-activation; E4M3), the allocation-free entry
   point and the host-buffer path report NM_OK: no range was missed;
 - their outputs are bit-identical to the normal library's (run here, in the
   parent) and match the oracle;
 - with the test hook lowering the TMEM limit below what the plan uses, the
   same dispatch reports NM_ERR_RANGE_CHECK (the checks do run) and still
   writes the same outputs; with the limit restored it reports NM_OK again.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for _p in (ROOT, HERE):
    if _p not in sys.path:
        sys.path.insert(0, _p)

from mlp_neural_gb300 import synth  # noqa: E402

N_ROWS = 152 * 128 * 3 + 77   # every CTA, three rounds, a ragged tail

# (name, dims, variant name, path): "infer" (nm_mlp_infer), "host"
# (nm_mlp_infer_host), "noalloc" (nm_mlp_infer_noalloc)
CASES = [
    ("page", synth.WORKLOADS["page"].dims, "NM_VARIANT_FUSED", "infer"),
    ("page-rowmajor", synth.WORKLOADS["page"].dims, "NM_VARIANT_ROWMAJOR_WEIGHTS", "infer"),
    ("page-scalar", synth.WORKLOADS["page"].dims, "NM_VARIANT_SCALAR_ACTIVATION", "infer"),
    ("page-paired", synth.WORKLOADS["page"].dims, "NM_VARIANT_PAIRED_TILES", "infer"),
    ("tiny", synth.WORKLOADS["tiny"].dims, "NM_VARIANT_FUSED", "infer"),
    ("wide", synth.WORKLOADS["wide"].dims, "NM_VARIANT_FUSED", "infer"),
    ("wide-scalar", synth.WORKLOADS["wide"].dims, "NM_VARIANT_SCALAR_ACTIVATION", "infer"),
    ("wide-fp8", synth.WORKLOADS["wide"].dims, "NM_VARIANT_FP8_WEIGHTS", "infer"),
    ("hetero", synth.WORKLOADS["hetero"].dims, "NM_VARIANT_FUSED", "infer"),
    ("hetero-fp8", synth.WORKLOADS["hetero"].dims, "NM_VARIANT_FP8_WEIGHTS", "infer"),
    ("k-tails", (80,) + (96,) * 8 + (16,), "NM_VARIANT_FUSED", "infer"),
    ("k-tails-fp8", (48, 96, 224, 32, 16), "NM_VARIANT_FP8_WEIGHTS", "infer"),
    ("streamed-deep", (64,) + (96,) * 15 + (16,), "NM_VARIANT_FUSED", "infer"),
    ("wide-256", (256, 256, 256, 16), "NM_VARIANT_FUSED", "infer"),
    ("wide-host", synth.WORKLOADS["wide"].dims, "NM_VARIANT_FUSED", "host"),
    ("page-noalloc", synth.WORKLOADS["page"].dims, "NM_VARIANT_FUSED", "noalloc"),
]
# dispatches repeated with the TMEM limit lowered by the test hook
LIMIT_CASES = ["page", "wide", "hetero-fp8"]


def _inputs(i, dims):
    return synth.small_net_inputs(dims, seed=500 + i, n=N_ROWS)


def _run_case(lib, dims, variant, path, W, b, x, check_limit=0):
    """One dispatch; returns (outputs as uint16, device status)."""
    import torch
    from gpu_util import make_net, to_dev, to_host
    n = x.shape[0]
    if path == "noalloc":
        out = torch.empty((n, dims[-1]), dtype=torch.float16, device="cuda")
        st = lib.infer_noalloc(dims, [to_dev(w) for w in W], [to_dev(v) for v in b], to_dev(x), out)
        torch.cuda.synchronize()
        return to_host(out), st
    m = make_net(dims, W, b)
    m.set_variant(getattr(lib, variant))
    if check_limit:
        m.set_test_check_limit(check_limit)
    if path == "host":
        m.set_host_chunk(8192)
        xh = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.float16).pin_memory()
        out = torch.empty((n, dims[-1]), dtype=torch.float16).pin_memory()
        m.infer_host(xh, out)
        torch.cuda.synchronize()
        y = out.view(torch.int16).numpy().view(np.uint16).copy()
    else:
        out = m.infer(to_dev(x))
        torch.cuda.synchronize()
        y = to_host(out)
    st = m.device_status()
    m.close()
    return y, st


def _child(out_dir):
    """Runs under NM_CHECKED=1: every case on the checking library."""
    import torch
    from gpu_util import nm
    lib = nm()
    assert lib.CHECKED and lib.checking_build(), "NM_CHECKED=1 did not load the checking build"
    torch.cuda.set_device(0)
    report = {"status": {}, "limited": {}}
    for i, (name, dims, variant, path) in enumerate(CASES):
        W, b, x = _inputs(i, dims)
        y, st = _run_case(lib, dims, variant, path, W, b, x)
        report["status"][name] = int(st)
        np.save(os.path.join(out_dir, f"{name}.npy"), y)
        if name in LIMIT_CASES:
            plan = lib.plan(dims, getattr(lib, variant))
            # below the plan's TMEM columns: the accumulator checks must fire
            y2, st2 = _run_case(lib, dims, variant, path, W, b, x, check_limit=16)
            y3, st3 = _run_case(lib, dims, variant, path, W, b, x)
            report["limited"][name] = {"status": int(st2), "same": bool(np.array_equal(y2, y)),
                                       "after": int(st3), "after_same": bool(np.array_equal(y3, y)),
                                       "tmem_columns": int(plan["tmem_columns"])}
    with open(os.path.join(out_dir, "report.json"), "w") as f:
        json.dump(report, f)


@pytest.mark.gpu
def test_checking_build_passes_and_matches_the_normal_build(orc, tmp_path):
    import torch
    from gpu_util import assert_close, nm
    from mlp_neural_gb300 import build
    lib = nm()
    if lib.CHECKED:
        pytest.skip("compares the checking build with the normal one: run without NM_CHECKED")
    assert not lib.checking_build()
    build.build(checked=True)
    env = dict(os.environ, NM_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), str(tmp_path)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    report = json.load(open(tmp_path / "report.json"))
    bad = {k: lib.status_str(v) for k, v in report["status"].items() if v != lib.NM_OK}
    assert not bad, f"checking build reported: {bad}"
    for name, rec in report["limited"].items():
        assert rec["status"] == lib.NM_ERR_RANGE_CHECK, (name, rec)
        assert rec["same"] and rec["after_same"], (name, rec)
        assert rec["after"] == lib.NM_OK, (name, rec)
    torch.cuda.set_device(0)
    for i, (name, dims, variant, path) in enumerate(CASES):
        W, b, x = _inputs(i, dims)
        y_chk = np.load(tmp_path / f"{name}.npy")
        y, st = _run_case(lib, dims, variant, path, W, b, x)
        assert st == lib.NM_OK, name
        assert np.array_equal(y_chk, y), f"{name}: checking build differs from the normal build"
        # the oracle on a sample of rows: the first 2,000 and the ragged last tile
        rows = np.r_[0:2000, N_ROWS - 205:N_ROWS]
        if variant == "NM_VARIANT_FP8_WEIGHTS":
            from test_gpu_fp8 import fp8_compare
            fp8_compare(y[rows], orc.forward_fp8(dims, W, b, x[rows]), name)
        else:
            assert_close(y[rows], orc.forward(dims, W, b, x[rows]), name)


if __name__ == "__main__":
    _child(sys.argv[1])
