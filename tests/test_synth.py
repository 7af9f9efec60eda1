"""Pins of the seeded input generator (CPU only)."""
import numpy as np

from mlp_neural_gb300 import synth


def test_splitmix64_published_vectors():
    # Reference outputs of SplitMix64 (Steele, Lea, Flood 2014; Vigna's
    # splitmix64.c) for seeds 0 and 1234567.
    assert [int(v) for v in synth.splitmix64(0, 0, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [int(v) for v in synth.splitmix64(1234567, 0, 2)] == [
        6457827717110365317, 3203168211198807973]


def test_counter_based_offsets():
    a = synth.splitmix64(9, 0, 100)
    b = synth.splitmix64(9, 37, 20)
    assert np.array_equal(a[37:57], b)


def test_net_params_ranges_and_order():
    dims = (48, 64, 16)
    W, b = synth.net_params(dims, seed=1)
    assert W[0].shape == (64, 48) and W[1].shape == (16, 64)
    w0 = W[0].view(np.float16).astype(np.float64)
    assert np.abs(w0).max() <= np.sqrt(6 / 48) * (1 + 2 ** -10)
    assert np.abs(b[1].view(np.float16).astype(np.float64)).max() <= 0.1 * (1 + 2 ** -10)
    # draw order: W_1 row-major first, so its first element is draw #1
    u = synth.uniform01(1, 0, 1)[0]
    a = np.sqrt(6 / 48)
    first = np.float16(np.float32(-a + 2 * a * u))
    assert W[0][0, 0] == first.view(np.uint16)
    # biases of layer 1 follow its 64*48 weights
    ub = synth.uniform01(1, 64 * 48, 1)[0]
    assert b[0][0] == np.float16(np.float32(-0.1 + 0.2 * ub)).view(np.uint16)


def test_inputs_follow_params_and_are_sliceable():
    w = synth.WORKLOADS["page"]
    x_all = synth.inputs(w, 0, 1000)
    x_mid = synth.inputs(w, 600, 50)
    assert np.array_equal(x_all[600:650], x_mid)
    u = synth.uniform01(w.seed, w.param_draws, 1)[0]
    assert x_all[0, 0] == np.float16(np.float32(-1 + 2 * u)).view(np.uint16)
    v = x_all.view(np.float16)
    assert np.abs(v).max() <= 1 and v.std() > 0.5


def test_normal_inputs_clipped():
    w = synth.WORKLOADS["hetero"]
    x = synth.inputs(w, 0, 20000).view(np.float16).astype(np.float64)
    assert np.abs(x).max() <= 4.0
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02


def test_workload_table():
    t = synth.WORKLOADS
    assert t["tiny"].n_evals == 65536 and t["page"].n_evals == 1048576
    assert t["ablation"].n_evals == 1048576 and t["wide"].n_evals == 16777216
    assert t["hetero"].n_evals == 4194304
    assert t["page"].flops_per_eval == 57344 and t["page"].hbm_bytes_per_eval == 128
    assert t["tiny"].flops_per_eval == 15360 and t["wide"].flops_per_eval == 217088
    assert t["hetero"].flops_per_eval == 337920
    assert all(w.n_layers == 8 for w in t.values())
