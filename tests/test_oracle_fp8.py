"""Pins of the oracle's narrow-precision variant (CPU only).

The reading (the pages name quantization as a pillar -- "Optimization
Techniques: Squeezing the Silicon", chapter introduction -- and stream narrow
weight codes through a TMA ring -- ninfer pull request #160 -- but fix no
format): layers 2..L multiply OCP E4M3 weights with E4M3 activations, layer
1 stays FP16, sums are FP32, biases FP16, every layer's result is rounded
once to FP16 and hidden layers apply the FP16 activation before the next
layer's E4M3 rounding.

Checked against things other than the oracle's own code:
 - E4M3 decoding of all 256 codes and RNE encoding of every finite FP16 value
   up to 448 against PyTorch's float8_e4m3fn conversion (a library routine);
 - saturation above 448 and NaN, from the satfinite reading;
 - the forward pass against a float64 brute force that quantizes with
   PyTorch's float8 cast and rounds with numpy's float16, on networks whose
   FP32 sums are exact (so the two must agree bit for bit), with layer-1
   weights that E4M3 cannot hold (a quantized first layer fails);
 - the E4M3 image layout against its 16-byte-chunk restatement and
   hand-computed sizes.
"""
import numpy as np
import pytest
import torch

from mlp_neural_gb300 import synth
from netgen import exact_fp8_net

SLOPE = np.float16(0.01)


def _torch_e4m3(v16: np.ndarray) -> np.ndarray:
    """FP16 values -> E4M3 -> float64 through PyTorch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(v16, dtype=np.float16))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_all_codes(orc):
    c = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_f32_array(c)
    ref = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.isnan(got).sum() == 2          # S.1111.111 only
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_every_fp16_in_range(orc):
    h = np.arange(65536, dtype=np.uint16)
    f = h.view(np.float16)
    got = orc.f16_to_e4m3_array(h)
    ref = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    fin = np.isfinite(f) & (np.abs(f.astype(np.float64)) <= 448.0)
    assert fin.sum() > 48000
    assert np.array_equal(got[fin], ref[fin])


def test_e4m3_encode_saturates_and_keeps_nan(orc):
    h = np.arange(65536, dtype=np.uint16)
    f = h.view(np.float16).astype(np.float64)
    got = orc.f16_to_e4m3_array(h)
    big = np.isfinite(f) & (np.abs(f) > 448.0) | np.isinf(f)
    assert np.all(got[big & (f > 0)] == 0x7E) and np.all(got[big & (f < 0)] == 0xFE)
    nan = np.isnan(f)
    assert np.all((got[nan] & 0x7F) == 0x7F)
    # ties go to even: 17 * 2^-4 is halfway between 1.0 (code 0x38) and
    # 1.125 (0x39) -> 0x38; 19 * 2^-4 halfway between 0x39 and 0x3A -> 0x3A
    assert orc.f16_to_e4m3_array(np.array([1.0625, 1.1875], np.float16).view(np.uint16)).tolist() == [0x38, 0x3A]


def _brute_fp8(dims, W, b, x):
    cur = x.view(np.float16).astype(np.float64)
    L = len(dims) - 1
    for l in range(L):
        w16 = W[l].view(np.float16)
        w = w16.astype(np.float64) if l == 0 else _torch_e4m3(w16)
        z = cur @ w.T + b[l].view(np.float16).astype(np.float64)
        h = z.astype(np.float16)                 # one RNE rounding to FP16
        if l < L - 1:
            h = np.maximum(h, h * SLOPE)         # FP16 product, exact in FP32
            cur = _torch_e4m3(h)                 # next layer reads E4M3
        else:
            return h.view(np.uint16)


@pytest.mark.parametrize("dims", [(32, 64, 32, 16), (64, 128, 128, 16), (48, 96, 64, 160, 32)])
def test_forward_fp8_against_brute_force(orc, dims):
    W, b = exact_fp8_net(dims, seed=sum(dims))
    rng = np.random.default_rng(7)
    x = (rng.integers(-255, 256, size=(300, dims[0])) * 2.0 ** -8).astype(np.float16).view(np.uint16)
    got = orc.forward_fp8(dims, W, b, x)
    ref = _brute_fp8(dims, W, b, x)
    assert np.array_equal(got, ref)
    # the narrow layers change the result: the FP16 pass differs somewhere
    assert not np.array_equal(got, orc.forward(dims, W, b, x))


def test_forward_fp8_close_to_fp16_on_a_random_network(orc):
    dims = synth.WORKLOADS["wide"].dims
    W, b, x = synth.small_net_inputs(dims, seed=3, n=512)
    y8 = orc.forward_fp8(dims, W, b, x).view(np.float16).astype(np.float64)
    y16 = orc.forward(dims, W, b, x).view(np.float16).astype(np.float64)
    rel = np.linalg.norm(y8 - y16) / np.linalg.norm(y16)
    assert 1e-3 < rel < 0.15, rel


def test_forward_fp8_rejects_one_layer(orc):
    W, b, x = synth.small_net_inputs((32, 16), seed=1, n=4)
    with pytest.raises(ValueError):
        orc.forward_fp8((32, 16), W, b, x)


def _segments8(K):
    segs, k0 = [], 0
    while K - k0 >= 128:
        segs.append((k0, 128)); k0 += 128
    if K - k0 >= 64:
        segs.append((k0, 64)); k0 += 64
    if K - k0 >= 32:
        segs.append((k0, 32)); k0 += 32
    assert k0 == K
    return segs


def _chunk_pos8(n, kk, w):
    """Byte offset of byte column kk of row n in a w-byte-wide segment: the
    16-byte chunk kk // 16 XORed with the row's place in its swizzle atom
    (128-byte rows: n % 8; 64-byte: (n // 2) % 4; 32-byte: (n // 4) % 2)."""
    c, e = kk // 16, kk % 16
    key = {128: n % 8, 64: (n // 2) % 4, 32: (n // 4) % 2}[w]
    return n * w + (c ^ key) * 16 + e


FP8_DIMS = [synth.WORKLOADS["wide"].dims, synth.WORKLOADS["hetero"].dims,
            (48, 96, 224, 32, 16), (64, 160, 16)]


@pytest.mark.parametrize("dims", FP8_DIMS)
def test_pack_fp8_matches_chunk_definition(orc, dims):
    W, b, _ = synth.small_net_inputs(dims, seed=8, n=1)
    region = orc.pack_fp8(dims, W)
    size, img = orc.fp8_layout(dims)
    expect = np.zeros(size, np.uint8)
    for l in range(1, len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        q = torch.from_numpy(W[l].view(np.float16).copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        off = img[l]
        assert off % 1024 == 0
        for k0, w in _segments8(K):
            off = (off + 1023) // 1024 * 1024
            for n in range(N):
                for kk in range(w):
                    expect[off + _chunk_pos8(n, kk, w)] = q[n, k0 + kk]
            off += N * w
        end = off
    assert end == size
    assert np.array_equal(region, expect)


def test_fp8_sizes(orc):
    # wide: six 128x128 images of 16 KiB and a 16x128 one of 2 KiB
    size, img = orc.fp8_layout(synth.WORKLOADS["wide"].dims)
    assert img == [None] + [16384 * i for i in range(7)] and size == 6 * 16384 + 2048
    # hetero: layers 2..8 hold 160,768 weights, every image a multiple of 1 KiB
    size, _ = orc.fp8_layout(synth.WORKLOADS["hetero"].dims)
    assert size == 168960 - 64 * 128


@pytest.mark.parametrize("dims", [(32, 16), (32, 48, 16), (64, 128, 80, 16)])
def test_fp8_layout_rejects(orc, dims):
    with pytest.raises(ValueError):
        orc.fp8_layout(dims)
