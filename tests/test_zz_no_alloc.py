"""nm_mlp_infer_noalloc: inference for callers that cannot allocate device
memory (for example code inside a host application that owns the device's
memory budget). It keeps its packed weights in a library-owned static device
array, so these tests check that two calls in a row -- on different networks,
so the second must not see the first's leftovers -- give the same outputs as
the handle-based nm_mlp_infer, within the parity tolerance.

This file is collected last on purpose, and each test works whether it runs
alone in a fresh process or after the other tests.
"""
import numpy as np
import pytest

from mlp_neural_gb300 import synth
from gpu_util import assert_close, make_net, nm, to_dev, to_host

pytestmark = pytest.mark.gpu


def _reference(dims, W, b, xd):
    import torch
    m = make_net(dims, W, b)
    out = m.infer(xd)
    torch.cuda.synchronize()
    assert m.device_status() == nm().NM_OK
    y = to_host(out)
    m.close()
    return y


def test_noalloc_matches_handle_path_two_calls_in_a_row():
    import torch
    lib = nm()
    cases = [(synth.WORKLOADS["page"].dims, 5000 + 77), (synth.WORKLOADS["tiny"].dims, 3 * 128 + 5)]
    for dims, n in cases:
        W, b, x = synth.small_net_inputs(dims, seed=n, n=n)
        Wd = [to_dev(w) for w in W]
        bd = [to_dev(v) for v in b]
        xd = to_dev(x)
        ref = _reference(dims, W, b, xd)
        out = torch.full((n, dims[-1]), float("nan"), dtype=torch.float16, device="cuda")
        st = lib.infer_noalloc(dims, Wd, bd, xd, out)
        assert st == lib.NM_OK, lib.status_str(st)
        assert_close(to_host(out), ref, f"noalloc dims={dims}")


def test_noalloc_rejects_oversized_network():
    import torch
    lib = nm()
    dims = (256,) * 10   # packed weights about 1.2 MB, beyond the 1 MiB scratch
    W = [torch.zeros((256, 256), dtype=torch.float16, device="cuda") for _ in range(9)]
    b = [torch.zeros(256, dtype=torch.float16, device="cuda") for _ in range(9)]
    x = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    out = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    assert lib.infer_noalloc(dims, W, b, x, out) == lib.NM_ERR_UNSUPPORTED
