"""Network generators shared by the oracle pins and the GPU tests (no tests
here)."""
import numpy as np


def exact_fp8_net(dims, seed):
    """A network whose FP32 sums are exact: every weight of layers >= 2 is
    E4M3 with exponent in [-4, -1]; layer-1 weights have 8 significant bits
    (E4M3 cannot hold most of them); biases are multiples of 2^-8 below 1/4."""
    rng = np.random.default_rng(seed)
    W, b = [], []
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        sgn = rng.choice([-1.0, 1.0], size=(N, K))
        if l == 0:
            v = sgn * rng.integers(128, 256, size=(N, K)) * 2.0 ** rng.integers(-12, -8, size=(N, K))
        else:
            v = sgn * (8 + rng.integers(0, 8, size=(N, K))) * 2.0 ** rng.integers(-7, -4, size=(N, K))
        W.append(v.astype(np.float16).view(np.uint16))
        b.append((rng.integers(-64, 64, size=N) * 2.0 ** -8).astype(np.float16).view(np.uint16))
    return W, b
