"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: packed weights bit-exact; outputs within |gpu - cpu| <= 1e-2 + 1e-2|cpu|
per element on random data; bit-exact wherever every FP32 partial sum is
exact (dyadic and signed-permutation networks, the activation on every finite
FP16 value); the two ablation variants bit-identical to the fused kernel.
"""
import numpy as np
import pytest

from mlp_neural_gb300 import synth
from gpu_util import assert_close, check_rows_parallel, make_net, nm, read_device, to_dev, to_host

pytestmark = pytest.mark.gpu

SMALL_DIMS = [
    synth.WORKLOADS["tiny"].dims,
    synth.WORKLOADS["page"].dims,
    (48, 80, 112, 16),
    (16, 16),
    (64, 128, 128, 32),
    (32, 48, 96, 208, 16),
    (256, 128, 16),      # 16 k-slabs in one layer (resident weights)
    (32,) * 17,          # the most layers a network may have
]
# Networks whose packed weights do not fit in shared memory: the kernel
# streams their weights (wide: 2 tile slots, heterogeneous: 1).
STREAMED_DIMS = [synth.WORKLOADS["wide"].dims, synth.WORKLOADS["hetero"].dims,
                 (48, 240, 208, 176, 16),    # 1 slot; K-segments of 64, 32 and 16
                 (80,) + (112,) * 8 + (16,),  # 2 slots; every K leaves a tail
                 (64,) + (96,) * 15 + (16,),  # 3 slots of 4 warps, 16 layers
                 (128, 128, 64, 128, 128, 128, 128, 64, 128, 16)]  # 3 slots, A split TMEM/smem
SENTINEL = 0x7E7E  # a NaN pattern the kernel never produces from finite data


def _run(m, x16, extra_rows=0, variant=None):
    import torch
    n = x16.shape[0]
    out = torch.full((n + extra_rows, m.dims[-1]), 0, dtype=torch.int16, device="cuda")
    out.fill_(np.int16(np.uint16(SENTINEL).view(np.int16)))
    out = out.view(torch.float16)
    if variant is not None:
        m.set_variant(variant)
    xd = to_dev(x16) if n else torch.empty((0, m.dims[0]), dtype=torch.float16, device="cuda")
    m.infer(xd, out[:n] if n else out[:0])
    torch.cuda.synchronize()
    assert m.device_status() == nm().NM_OK
    y = to_host(out)
    assert (y[n:] == SENTINEL).all(), "rows beyond n were written"
    return y[:n]


@pytest.mark.parametrize("dims", SMALL_DIMS + [synth.WORKLOADS["hetero"].dims,
                                               synth.WORKLOADS["wide"].dims])
def test_pack_bit_exact(orc, dims):
    W, b, _ = synth.small_net_inputs(dims, seed=21, n=1)
    m = make_net(dims, W, b)
    ref = orc.pack(dims, W, b)
    assert m.packed_size() == ref.size
    got = read_device(m.packed_blob(), ref.size)
    assert np.array_equal(got, ref)
    # unpack on the device restores the canonical weights
    import torch
    W2 = [torch.zeros_like(to_dev(w)) for w in W]
    b2 = [torch.zeros_like(to_dev(v)) for v in b]
    m.unpack_weights(W2, b2)
    torch.cuda.synchronize()
    for l in range(len(W)):
        assert np.array_equal(to_host(W2[l]), W[l]) and np.array_equal(to_host(b2[l]), b[l])


@pytest.mark.parametrize("dims", SMALL_DIMS + STREAMED_DIMS)
@pytest.mark.parametrize("n", [1, 127, 128, 129, 255, 4097])
def test_infer_matches_oracle(orc, dims, n):
    W, b, x = synth.small_net_inputs(dims, seed=n + dims[0], n=n)
    m = make_net(dims, W, b)
    y = _run(m, x, extra_rows=300)
    assert_close(y, orc.forward(dims, W, b, x), f"dims={dims} n={n}")


def test_infer_many_tiles_ragged(orc):
    dims = synth.WORKLOADS["page"].dims
    n = 152 * 128 * 3 + 77   # several tiles per CTA and a ragged tail
    W, b, x = synth.small_net_inputs(dims, seed=99, n=n)
    m = make_net(dims, W, b)
    y = _run(m, x, extra_rows=129)
    assert_close(y, orc.forward(dims, W, b, x), "many tiles")


def _dyadic_net(dims, seed, n):
    rng = np.random.default_rng(seed)
    W, b = [], []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        w = np.zeros((N, K), np.float16)
        for r in range(N):
            w[r, rng.choice(K, size=4, replace=False)] = 0.25
        W.append(w.view(np.uint16))
        b.append((rng.integers(1, 9, size=N) / 64.0).astype(np.float16).view(np.uint16))
    x = (rng.integers(0, 9, size=(n, dims[0])) / 8.0).astype(np.float16).view(np.uint16)
    return W, b, x


@pytest.mark.parametrize("dims", SMALL_DIMS + STREAMED_DIMS)
def test_dyadic_networks_bit_exact(orc, dims):
    W, b, x = _dyadic_net(dims, seed=len(dims) * 7 + dims[-2], n=1000)
    m = make_net(dims, W, b)
    assert np.array_equal(_run(m, x), orc.forward(dims, W, b, x))


@pytest.mark.parametrize("dims", [(32,) * 9, (64,) * 9, (128, 128, 64), (48, 48, 48)])
def test_signed_permutation_networks_bit_exact(orc, dims):
    rng = np.random.default_rng(sum(dims))
    W, b = [], []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        w = np.zeros((N, K), np.float16)
        w[np.arange(N), rng.permutation(K)[:N]] = rng.choice([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0], size=N)
        W.append(w.view(np.uint16))
        b.append(np.zeros(N, np.uint16))
    x = rng.uniform(-1, 1, size=(777, dims[0])).astype(np.float16).view(np.uint16)
    m = make_net(dims, W, b)
    assert np.array_equal(_run(m, x), orc.forward(dims, W, b, x))


@pytest.mark.parametrize("variant", [0, 2])
def test_activation_on_every_finite_fp16_value(orc, variant):
    # Two identity layers of width 16: the first applies the activation to
    # the FP16 value it was given, the second passes it through. Every
    # finite FP16 pattern appears once as an input element.
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    pats = pats[(pats & 0x7C00) != 0x7C00]
    x = pats.reshape(-1, 16)
    eye = np.eye(16, dtype=np.float16).view(np.uint16)
    dims = (16, 16, 16)
    W, b = [eye, eye], [np.zeros(16, np.uint16)] * 2
    m = make_net(dims, W, b)
    y = _run(m, x, variant=variant)
    assert np.array_equal(y, orc.forward(dims, W, b, x))


@pytest.mark.parametrize("dims", [synth.WORKLOADS["tiny"].dims, synth.WORKLOADS["page"].dims,
                                  (48, 80, 112, 16)])
def test_ablation_variants_bit_identical(dims):
    W, b, x = synth.small_net_inputs(dims, seed=5, n=5000)
    m = make_net(dims, W, b)
    y0 = _run(m, x, variant=0)
    y1 = _run(m, x, variant=1)
    y2 = _run(m, x, variant=2)
    assert np.array_equal(y0, y1) and np.array_equal(y0, y2)


@pytest.mark.parametrize("dims", [synth.WORKLOADS["tiny"].dims, synth.WORKLOADS["page"].dims,
                                  (48, 80, 112, 16), (64, 128, 128, 32)])
@pytest.mark.parametrize("n", [5000, 152 * 128 * 6 + 333])
def test_paired_tiles_variant_bit_identical(dims, n):
    # two tile regions per issuing warp, including CTAs whose last round
    # fills only part of a pair
    W, b, x = synth.small_net_inputs(dims, seed=9, n=n)
    m = make_net(dims, W, b)
    assert np.array_equal(_run(m, x, variant=0), _run(m, x, variant=3))


@pytest.mark.parametrize("dims", STREAMED_DIMS)
def test_streamed_weights_scalar_activation_bit_identical(dims):
    W, b, x = synth.small_net_inputs(dims, seed=8, n=3000)
    m = make_net(dims, W, b)
    assert np.array_equal(_run(m, x, variant=0), _run(m, x, variant=2))


def test_empty_batch_and_argument_errors():
    lib = nm()
    dims = (32, 16)
    W, b, x = synth.small_net_inputs(dims, seed=1, n=4)
    m = lib.MLP(dims)
    xd = to_dev(x)
    import torch
    out = torch.empty((4, 16), dtype=torch.float16, device="cuda")
    assert m.infer_raw(xd.data_ptr(), 4, out.data_ptr()) == lib.NM_ERR_NOT_PACKED
    m.pack_weights([to_dev(w) for w in W], [to_dev(v) for v in b])
    assert m.infer_raw(xd.data_ptr(), 0, out.data_ptr()) == lib.NM_OK
    assert m.infer_raw(xd.data_ptr(), -1, out.data_ptr()) == lib.NM_ERR_INVALID_ARG
    assert m.infer_raw(0, 4, out.data_ptr()) == lib.NM_ERR_INVALID_ARG
    assert m.infer_raw(xd.data_ptr() + 2, 3, out.data_ptr()) == lib.NM_ERR_INVALID_ARG
    assert m.infer_raw(xd.data_ptr(), 4, out.data_ptr()) == lib.NM_OK
    assert m.device_status() == lib.NM_OK


def test_wait_limit_gives_up_cleanly(orc):
    # Every CTA first waits on a barrier nothing signals; after the 1 ms wait
    # limit the kernel must report NM_ERR_TIMEOUT, drain its copies, free its
    # tensor memory and leave the context usable for the next call.
    lib = nm()
    dims = synth.WORKLOADS["page"].dims
    W, b, x = synth.small_net_inputs(dims, seed=3, n=128 * 600)
    m = make_net(dims, W, b)
    m.set_wait_limit(1_000_000)
    m.set_test_stall(True)
    import torch
    xd = to_dev(x)
    out = torch.empty((x.shape[0], dims[-1]), dtype=torch.float16, device="cuda")
    for variant in (0, 1, 2):
        m.set_variant(variant)
        assert m.infer_raw(xd.data_ptr(), x.shape[0], out.data_ptr()) == lib.NM_OK
        assert m.device_status() == lib.NM_ERR_TIMEOUT
        assert m.device_status() == lib.NM_OK  # the status word was cleared
    m.set_test_stall(False)
    m.set_wait_limit(2_000_000_000)
    m.set_variant(0)
    y = _run(m, x[:1000])
    assert_close(y, orc.forward(dims, W, b, x[:1000]), "after give-up")


def _full_workload(orc, name, variants=(0,)):
    import torch
    w = synth.WORKLOADS[name]
    W, b = synth.net_params(w.dims, w.seed)
    xu = synth.inputs(w)
    m = make_net(w.dims, W, b)
    xd = to_dev(xu)
    if w.repeats > 1:
        xd = xd.repeat(w.repeats, 1)
    n = xd.shape[0]
    ref = orc.forward(w.dims, W, b, xu)
    outs = []
    for v in variants:
        m.set_variant(v)
        out = torch.empty((n, w.dims[-1]), dtype=torch.float16, device="cuda")
        m.infer(xd, out)
        torch.cuda.synchronize()
        assert m.device_status() == nm().NM_OK
        y = to_host(out).reshape(w.repeats, w.n_unique, w.dims[-1])
        for r in range(1, w.repeats):
            assert np.array_equal(y[r], y[0]), f"repeat {r} differs"
        assert_close(y[0], ref, name)
        outs.append(y[0])
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_full_tiny(orc):
    _full_workload(orc, "tiny")


def test_full_page(orc):
    _full_workload(orc, "page")


def test_full_ablation_all_variants(orc):
    _full_workload(orc, "ablation", variants=(0, 1, 2))


def test_full_tiny_ablation_all_variants(orc):
    """The ablations on the tiny network: its 65,536 inputs each evaluated 16
    times, the three variants bit-identical and within tolerance of the
    oracle."""
    _full_workload(orc, "tiny_ablation", variants=(0, 1, 2))


def _full_every_row(orc, name):
    """The full workload in one dispatch; every output row is compared with
    the oracle (run over all host cores)."""
    import time
    import torch
    w = synth.WORKLOADS[name]
    W, b = synth.net_params(w.dims, w.seed)
    x = synth.inputs(w)
    m = make_net(w.dims, W, b)
    xd = to_dev(x)
    out = torch.empty((w.n_evals, w.dims[-1]), dtype=torch.float16, device="cuda")
    m.infer(xd, out)
    torch.cuda.synchronize()
    assert m.device_status() == nm().NM_OK
    y = to_host(out)
    del xd, out
    m.close()
    t0 = time.time()
    rows, emax, threads = check_rows_parallel(orc, w.dims, W, b, x, y)
    print(f"{name}: {rows:,} rows checked against the oracle on {threads} threads in "
          f"{time.time() - t0:.0f} s, max |gpu-cpu| = {emax:.3g}")


def test_full_wide_every_row(orc):
    _full_every_row(orc, "wide")


def test_full_hetero_every_row(orc):
    _full_every_row(orc, "hetero")


def test_many_rotating_buffer_sets(orc):
    """More distinct (in, out) buffer pairs than the handle caches tensor maps
    for: every dispatch must still read its own input and write its own
    output."""
    import torch
    dims = (32, 48, 16)
    n = 300
    W, b, _ = synth.small_net_inputs(dims, seed=5, n=1)
    m = make_net(dims, W, b)
    sets = []
    for i in range(20):
        _, _, x = synth.small_net_inputs(dims, seed=100 + i, n=n)
        sets.append((x, to_dev(x), torch.empty((n, dims[-1]), dtype=torch.float16, device="cuda")))
    for rep in range(2):
        for x, xd, od in sets:
            m.infer(xd, od)
    torch.cuda.synchronize()
    assert m.device_status() == nm().NM_OK
    for x, xd, od in sets:
        assert_close(to_host(od), orc.forward(dims, W, b, x))
    m.close()


def test_infer_captured_in_cuda_graph(orc):
    """nm_mlp_infer is capturable: a graph replays the dispatch on new input
    contents written into the same buffers."""
    import torch
    dims = synth.WORKLOADS["page"].dims
    n = 1000
    W, b, x1 = synth.small_net_inputs(dims, seed=21, n=n)
    _, _, x2 = synth.small_net_inputs(dims, seed=22, n=n)
    m = make_net(dims, W, b)
    xd = to_dev(x1)
    od = torch.empty((n, dims[-1]), dtype=torch.float16, device="cuda")
    m.infer(xd, od)  # one eager dispatch first (one-time launch set-up)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        m.infer(xd, od, stream=side)
    for x in (x1, x2):
        xd.copy_(to_dev(x))
        od.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(to_host(od), orc.forward(dims, W, b, x))
    assert m.device_status() == nm().NM_OK
    m.close()


def _signed_permutation_net(dims, rng, scales):
    W, b = [], []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        w = np.zeros((N, K), np.float16)
        w[np.arange(N), rng.permutation(K)[:N]] = rng.choice(scales, size=N)
        W.append(w.view(np.uint16))
        b.append(np.zeros(N, np.uint16))
    return W, b


@pytest.mark.parametrize("dims", [(64,) * 9, (128,) * 9])
def test_back_to_back_dispatches_chain_through_buffers(orc, dims):
    """Dispatches queued back to back on one stream overlap only their
    prologues: each reads its input after the previous dispatch wrote it, and
    writes its output after the previous dispatch read it. The network is
    exact (one product per output), so every link of the chain is bit-exact
    whatever the others computed."""
    import torch
    rng = np.random.default_rng(sum(dims) + 5)
    W, b = _signed_permutation_net(dims, rng, [-1.0, -0.5, 0.5, 1.0])
    n = 152 * 128 * 2 + 77  # several tiles per CTA and a ragged tail
    x = rng.uniform(-1, 1, size=(n, dims[0])).astype(np.float16).view(np.uint16)
    m = make_net(dims, W, b)
    X = to_dev(x)
    A = torch.empty((n, dims[-1]), dtype=torch.float16, device="cuda")
    B = torch.empty_like(A)
    m.infer(X, A)  # y1
    m.infer(A, B)  # y2 = f(y1): reads what the previous dispatch wrote
    m.infer(B, A)  # y3 = f(y2): overwrites what the previous dispatch read
    m.infer(A, X)  # y4 = f(y3)
    torch.cuda.synchronize()
    assert m.device_status() == nm().NM_OK
    y1 = orc.forward(dims, W, b, x)
    y2 = orc.forward(dims, W, b, y1)
    y3 = orc.forward(dims, W, b, y2)
    y4 = orc.forward(dims, W, b, y3)
    assert np.array_equal(to_host(B), y2)
    assert np.array_equal(to_host(A), y3)
    assert np.array_equal(to_host(X), y4)
    m.close()


@pytest.mark.parametrize("dims", [synth.WORKLOADS["page"].dims, synth.WORKLOADS["wide"].dims])
def test_repack_between_dispatches_on_one_stream(orc, dims):
    """A dispatch queued right after a repack on the same stream uses the new
    weights, and the one queued before it the old ones."""
    import torch
    W1, b1, x = synth.small_net_inputs(dims, seed=41, n=3000)
    W2, b2, _ = synth.small_net_inputs(dims, seed=42, n=1)
    m = make_net(dims, W1, b1)
    dev1 = ([to_dev(w) for w in W1], [to_dev(v) for v in b1])
    dev2 = ([to_dev(w) for w in W2], [to_dev(v) for v in b2])
    xd = to_dev(x)
    outs = [torch.empty((x.shape[0], dims[-1]), dtype=torch.float16, device="cuda")
            for _ in range(4)]
    torch.cuda.synchronize()
    m.infer(xd, outs[0])
    m.pack_weights(*dev2)
    m.infer(xd, outs[1])
    m.infer(xd, outs[2])
    m.pack_weights(*dev1)
    m.infer(xd, outs[3])
    torch.cuda.synchronize()
    assert m.device_status() == nm().NM_OK
    y = [to_host(o) for o in outs]
    assert_close(y[0], orc.forward(dims, W1, b1, x), "before the repack")
    assert_close(y[1], orc.forward(dims, W2, b2, x), "right after the repack")
    assert np.array_equal(y[2], y[1])
    assert np.array_equal(y[3], y[0])
    m.close()


def test_two_handles_on_two_streams(orc):
    """Two networks dispatched concurrently on two streams do not disturb
    each other."""
    import torch
    nets = []
    for seed, dims in ((31, (32, 64, 16)), (32, synth.WORKLOADS["page"].dims)):
        W, b, x = synth.small_net_inputs(dims, seed=seed, n=5000)
        m = make_net(dims, W, b)
        out = torch.empty((5000, dims[-1]), dtype=torch.float16, device="cuda")
        nets.append((dims, W, b, x, m, to_dev(x), out, torch.cuda.Stream()))
    torch.cuda.synchronize()
    for _ in range(3):
        for dims, W, b, x, m, xd, out, st in nets:
            m.infer(xd, out, stream=st)
    torch.cuda.synchronize()
    for dims, W, b, x, m, xd, out, st in nets:
        assert m.device_status() == nm().NM_OK
        assert_close(to_host(out), orc.forward(dims, W, b, x))
        m.close()
