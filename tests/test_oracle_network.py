"""Pins of the oracle's network evaluation (CPU only).

Each expected value below comes from something other than the oracle:
 - identity and signed-permutation networks: every output is one input times
   a power of two, so it is exact, and the chain reduces to repeated
   activation, computed here with numpy's float16 arithmetic;
 - a one-layer network: a float64 brute-force dot product, within the
   rounding bound of an FP32 k-order sum plus one FP16 rounding;
 - dyadic networks whose every partial sum is exact in FP32: the result does
   not depend on summation order, so a numpy float64 matmul per layer with a
   float16 rounding after it must agree bit for bit;
 - random networks: numpy float64 per-layer evaluation with FP16 rounding
   between layers, within the parity tolerance.
"""
import numpy as np
import pytest

from mlp_neural_gb300 import synth

SLOPE = np.float16(0.01)
CONFIG_DIMS = [w.dims for w in synth.WORKLOADS.values()]


def np_leaky(h16):
    return np.where(h16 < 0, h16 * SLOPE, h16).astype(np.float16)


def np_forward_f64(dims, W, b, x):
    """float64 matmul per layer, rounded to float16 after each layer."""
    h = x.view(np.float16).astype(np.float64)
    L = len(dims) - 1
    for l in range(L):
        w = W[l].view(np.float16).astype(np.float64)
        bb = b[l].view(np.float16).astype(np.float64)
        v = (h @ w.T + bb).astype(np.float16)
        if l < L - 1:
            v = np_leaky(v)
        h = v.astype(np.float64)
    return h.astype(np.float16).view(np.uint16)


def test_identity_network_is_repeated_activation(orc):
    dims = [32] * 9
    L = 8
    eye = np.eye(32, dtype=np.float16).view(np.uint16)
    W = [eye.copy() for _ in range(L)]
    b = [np.zeros(32, np.uint16) for _ in range(L)]
    W0, b0, x = synth.small_net_inputs(dims, seed=7, n=300)
    x = np.concatenate([x, np.array([[0x8000, 0x0001, 0x8001, 0x7BFF, 0xFBFF, 0x3C00, 0xBC00,
                                      0x0400, 0x8400] + [0] * 23], dtype=np.uint16)])
    y = orc.forward(dims, W, b, x)
    # Each layer is a dot product that starts from +0 and adds a +0 bias, so
    # a -0 input comes out as +0 (IEEE: -0 + +0 = +0); then the activation.
    h = x.view(np.float16)
    for l in range(L):
        h = (h.astype(np.float32) + np.float32(0)).astype(np.float16)
        if l < L - 1:
            h = np_leaky(h)
    assert np.array_equal(y, h.view(np.uint16))


@pytest.mark.parametrize("dims", [(32,) * 9, (64,) * 9, (128, 128, 128, 128)])
def test_signed_permutation_network(orc, dims):
    rng = np.random.default_rng(sum(dims))
    L = len(dims) - 1
    W, b = [], []
    d = dims[0]
    perms, scales = [], []
    for _ in range(L):
        p = rng.permutation(d)
        s = rng.choice([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0], size=d)
        w = np.zeros((d, d), np.float16)
        w[np.arange(d), p] = s
        W.append(w.view(np.uint16))
        b.append(np.zeros(d, np.uint16))
        perms.append(p)
        scales.append(s.astype(np.float16))
    x = rng.uniform(-1, 1, size=(257, d)).astype(np.float16)
    y = orc.forward(dims, W, b, x.view(np.uint16))
    h = x
    for l in range(L):
        # The FP32 product is exact and non-zero for any non-zero input; the
        # +0 start of the sum and the +0 bias turn a -0 product into +0; the
        # value is rounded to FP16 once, after the bias.
        prod = h.astype(np.float32)[:, perms[l]] * scales[l].astype(np.float32)
        h = (prod + np.float32(0)).astype(np.float16)
        if l < L - 1:
            h = np_leaky(h)
    assert np.array_equal(y, h.view(np.uint16))


def _ulp16(v):
    v = np.maximum(np.abs(v), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(v)) - 10)


@pytest.mark.parametrize("K,N", [(16, 16), (48, 32), (64, 16), (256, 64)])
def test_one_layer_matches_brute_force(orc, K, N):
    W, b, x = synth.small_net_inputs((K, N), seed=K * 1000 + N, n=2000)
    y = orc.forward((K, N), W, b, x).view(np.float16).astype(np.float64)
    xf = x.view(np.float16).astype(np.float64)
    wf = W[0].view(np.float16).astype(np.float64)
    bf = b[0].view(np.float16).astype(np.float64)
    exact = xf @ wf.T + bf
    mag = np.abs(xf) @ np.abs(wf).T + np.abs(bf)
    err32 = (K + 1) * 2.0 ** -24 * mag * 1.01
    bound = 0.5 * _ulp16(np.abs(exact) + err32) + err32
    assert np.all(np.abs(y - exact) <= bound)
    # and in the overwhelming majority of cases it is the rounded exact value
    same = (y == exact.astype(np.float16).astype(np.float64)).mean()
    assert same > 0.99


def _dyadic_net(dims, seed, n):
    """Non-negative dyadic network: inputs k/8, four weights of 1/4 per row,
    biases k/64 (k = 1..8). Every value stays in [1/64, 2] after layer 1, so
    each FP32 partial sum is exact and summation order cannot matter."""
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


@pytest.mark.parametrize("dims", CONFIG_DIMS)
def test_dyadic_network_is_order_independent(orc, dims):
    W, b, x = _dyadic_net(dims, seed=len(dims) + dims[0], n=300)
    y = orc.forward(dims, W, b, x)
    assert np.array_equal(y, np_forward_f64(dims, W, b, x))


@pytest.mark.parametrize("dims", CONFIG_DIMS + [(48, 80, 112, 16)])
def test_random_network_vs_float64(orc, dims):
    W, b, x = synth.small_net_inputs(dims, seed=11, n=400)
    y = orc.forward(dims, W, b, x).view(np.float16).astype(np.float64)
    ref = np_forward_f64(dims, W, b, x).view(np.float16).astype(np.float64)
    assert np.all(np.abs(y - ref) <= 1e-2 + 1e-2 * np.abs(ref))


def test_forward_rejects_bad_dims(orc):
    with pytest.raises(ValueError):
        orc.forward((32, 0), [np.zeros((0, 32), np.uint16)], [np.zeros(0, np.uint16)],
                    np.zeros((1, 32), np.uint16))


def test_forward_empty_batch(orc):
    W, b, _ = synth.small_net_inputs((32, 16), seed=1, n=1)
    y = orc.forward((32, 16), W, b, np.zeros((0, 32), np.uint16))
    assert y.shape == (0, 16)
