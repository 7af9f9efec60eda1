"""nm_mlp_infer_noalloc: inference for callers that cannot allocate device
memory (for example code inside a host application that owns the device's
memory budget). It keeps its packed weights in a library-owned static device
array, so these tests check that calls in a row -- on different networks, so
a later call must not see an earlier one's leftovers -- give the same outputs
as the handle-based nm_mlp_infer (bit for bit: both run the same kernel on
the same packed weights) and match the oracle within the parity tolerance.
One network is wide enough that its weights do not fit in shared memory, so
the kernel streams them out of the static array for the whole dispatch.

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


def test_noalloc_matches_handle_path_calls_in_a_row(orc):
    import torch
    lib = nm()
    cases = [(synth.WORKLOADS["page"].dims, 5000 + 77),
             (synth.WORKLOADS["tiny"].dims, 3 * 128 + 5),
             (synth.WORKLOADS["wide"].dims, 5000 + 13),   # streamed weights, 217 KB packed
             (synth.WORKLOADS["page"].dims, 1000)]
    for dims, n in cases:
        W, b, x = synth.small_net_inputs(dims, seed=n, n=n)
        Wd = [to_dev(w) for w in W]
        bd = [to_dev(v) for v in b]
        xd = to_dev(x)
        ref = _reference(dims, W, b, xd)
        out = torch.full((n, dims[-1]), float("nan"), dtype=torch.float16, device="cuda")
        st = lib.infer_noalloc(dims, Wd, bd, xd, out)
        assert st == lib.NM_OK, lib.status_str(st)
        got = to_host(out)
        assert np.array_equal(got, ref), f"noalloc differs from nm_mlp_infer, dims={dims}"
        assert_close(got, orc.forward(dims, W, b, x), f"noalloc dims={dims}")


def test_noalloc_rejects_oversized_network():
    import torch
    lib = nm()
    dims = (256,) * 10   # packed weights about 1.2 MB, beyond the 1 MiB scratch
    W = [torch.zeros((256, 256), dtype=torch.float16, device="cuda") for _ in range(9)]
    b = [torch.zeros(256, dtype=torch.float16, device="cuda") for _ in range(9)]
    x = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    out = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    assert lib.infer_noalloc(dims, W, b, x, out) == lib.NM_ERR_UNSUPPORTED


def test_noalloc_refuses_a_capturing_stream():
    """The call synchronises its stream, which graph capture forbids, so it
    answers NM_ERR_UNSUPPORTED before enqueuing anything; the capture stays
    valid and the stream usable."""
    import torch
    lib = nm()
    dims = synth.WORKLOADS["tiny"].dims
    W, b, x = synth.small_net_inputs(dims, seed=3, n=256)
    Wd = [to_dev(w) for w in W]
    bd = [to_dev(v) for v in b]
    xd = to_dev(x)
    out = torch.zeros((256, dims[-1]), dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        st = lib.infer_noalloc(dims, Wd, bd, xd, out, stream=side)
        out.add_(0)  # one captured op, so the graph is not empty
    assert st == lib.NM_ERR_UNSUPPORTED
    g.replay()
    torch.cuda.synchronize()
    assert lib.infer_noalloc(dims, Wd, bd, xd, out) == lib.NM_OK
