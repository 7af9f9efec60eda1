"""nm_mlp_infer_host: inputs and outputs in host memory, processed in chunks
on the handle's own streams. The kernel and the tile boundaries are those of
nm_mlp_infer (chunks are whole tiles), so the outputs must be bit-identical to
the device-buffer path on the same rows; the device path itself is checked
against the oracle elsewhere, and here once more on a sample."""
import numpy as np
import pytest

from mlp_neural_gb300 import synth
from gpu_util import assert_close, make_net, nm, to_dev, to_host

pytestmark = pytest.mark.gpu


def _host16(a16: np.ndarray, pinned: bool):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a16).view(np.int16)).view(torch.float16)
    return t.pin_memory() if pinned else t.clone()


def _device_path(m, x16):
    import torch
    out = m.infer(to_dev(x16))
    torch.cuda.synchronize()
    return to_host(out)


@pytest.mark.parametrize("dims", [synth.WORKLOADS["page"].dims, (32, 64, 16), (64, 128, 256, 16)])
@pytest.mark.parametrize("n,chunk", [(1, 256), (129, 256), (1000, 256), (1000, 128), (4097, 1024)])
def test_host_path_bit_identical_to_device_path(dims, n, chunk):
    import torch
    W, b, x = synth.small_net_inputs(dims, seed=n + chunk, n=n)
    m = make_net(dims, W, b)
    m.set_host_chunk(chunk)
    ref = _device_path(m, x)
    for pinned in (True, False):
        xh = _host16(x, pinned)
        out = torch.full((n, dims[-1]), float("nan"), dtype=torch.float16)
        if pinned:
            out = out.pin_memory()
        m.infer_host(xh, out)
        torch.cuda.current_stream().synchronize()
        got = out.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, ref), (dims, n, chunk, pinned)
    assert m.device_status() == nm().NM_OK
    m.close()


def test_host_path_default_chunk_many_chunks_and_oracle_sample(orc):
    import torch
    dims = synth.WORKLOADS["page"].dims
    n = 3 * 131072 + 1000  # the default chunk for d0 = 48 is 131,072 rows
    W, b, x = synth.small_net_inputs(dims, seed=11, n=n)
    m = make_net(dims, W, b)
    ref = _device_path(m, x)
    out = m.infer_host(_host16(x, True))
    torch.cuda.current_stream().synchronize()
    got = out.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    rows = np.r_[0:64, 131072 - 3:131072 + 3, n - 64:n]
    expect = orc.forward(dims, W, b, x[rows])
    assert_close(got[rows], expect)
    m.close()


def test_host_path_two_calls_reuse_the_pipeline():
    import torch
    dims = (32, 32, 32, 16)
    m = None
    outs, refs = [], []
    for seed in (1, 2):
        W, b, x = synth.small_net_inputs(dims, seed=seed, n=3000)
        if m is None:
            m = make_net(dims, W, b)
            m.set_host_chunk(512)
        else:
            m.pack_weights([to_dev(w) for w in W], [to_dev(v) for v in b])
        refs.append(_device_path(m, x))
        outs.append(m.infer_host(_host16(x, True)))
    torch.cuda.current_stream().synchronize()
    # the second call's weights replaced the first's only after the first
    # call's work: both results hold
    for o, r in zip(outs, refs):
        assert np.array_equal(o.view(torch.int16).numpy().view(np.uint16), r)
    m.close()


def test_host_path_argument_errors():
    import torch
    lib = nm()
    dims = (32, 16)
    W, b, x = synth.small_net_inputs(dims, seed=3, n=4)
    m = lib.MLP(dims)
    xh = _host16(x, False)
    out = torch.empty((4, 16), dtype=torch.float16)
    assert m.infer_host_raw(xh.data_ptr(), 4, out.data_ptr()) == lib.NM_ERR_NOT_PACKED
    m.pack_weights([to_dev(w) for w in W], [to_dev(v) for v in b])
    assert m.infer_host_raw(xh.data_ptr(), 0, out.data_ptr()) == lib.NM_OK
    assert m.infer_host_raw(0, 4, out.data_ptr()) == lib.NM_ERR_INVALID_ARG
    assert m.infer_host_raw(xh.data_ptr(), -1, out.data_ptr()) == lib.NM_ERR_INVALID_ARG
    for bad in (100, 127, 1 << 21, -128):
        with pytest.raises(lib.NmError):
            m.set_host_chunk(bad)
    m.set_host_chunk(0)
    m.close()
