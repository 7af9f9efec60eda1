"""Pins of the oracle's reference packer (CPU only).

The packed blob is this library's device-private weight layout (the pages'
"Row-major versus InferencingOptimal weights": a one-time conversion that
changes neither the network nor the activation). Its definition is written
out in the oracle; here it is checked against:
 - invertibility: unpack(pack(W, b)) == (W, b) bit for bit;
 - permutation: every weight and bias bit lands exactly once, padding is zero;
 - the 128-, 64- and 32-byte shared-memory swizzle patterns of the Blackwell
   TMA / UMMA K-major layouts, restated here in their 16-byte-chunk form
   (_chunk_pos), a different expression from the oracle's address XOR;
 - hand-computed blob sizes.
"""
import numpy as np
import pytest

from mlp_neural_gb300 import synth

CONFIG_DIMS = [w.dims for w in synth.WORKLOADS.values()]
ODD_DIMS = [(48, 80, 112, 16), (16, 16), (240, 16, 48, 256), (96, 208, 32)]


def _segments(K):
    segs, k0 = [], 0
    while K - k0 >= 64:
        segs.append((k0, 64)); k0 += 64
    if K - k0 >= 32:
        segs.append((k0, 32)); k0 += 32
    if K - k0 >= 16:
        segs.append((k0, 16)); k0 += 16
    assert k0 == K
    return segs


def _chunk_pos(n, kk, w):
    """Byte offset of element (row n, column kk within a w-wide segment).

    Rows are 2w bytes. The 16-byte chunk index c = kk // 8 is XORed with the
    row's position inside its 1024/512/256-byte swizzle atom:
      128-byte swizzle (w=64): c ^ (n % 8)
       64-byte swizzle (w=32): c ^ ((n // 2) % 4)
       32-byte swizzle (w=16): c ^ ((n // 4) % 2)
    """
    c, e = kk // 8, kk % 8
    key = {64: n % 8, 32: (n // 2) % 4, 16: (n // 4) % 2}[w]
    return n * 2 * w + (c ^ key) * 16 + e * 2


@pytest.mark.parametrize("dims", CONFIG_DIMS + ODD_DIMS)
def test_pack_roundtrip(orc, dims):
    W, b, _ = synth.small_net_inputs(dims, seed=5, n=1)
    blob = orc.pack(dims, W, b)
    W2, b2 = orc.unpack(dims, blob)
    for l in range(len(dims) - 1):
        assert np.array_equal(W[l], W2[l])
        assert np.array_equal(b[l], b2[l])


@pytest.mark.parametrize("dims", CONFIG_DIMS + ODD_DIMS)
def test_pack_matches_chunk_swizzle_definition(orc, dims):
    W, b, _ = synth.small_net_inputs(dims, seed=6, n=1)
    blob = orc.pack(dims, W, b)
    size, img, boff = orc.packed_layout(dims)
    words = blob.view(np.uint16)
    expect = np.zeros(size, np.uint8)
    ew = expect.view(np.uint16)
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        off = img[l]
        assert off % 1024 == 0
        for k0, w in _segments(K):
            off = (off + 1023) // 1024 * 1024
            for n in range(N):
                for kk in range(w):
                    ew[(off + _chunk_pos(n, kk, w)) // 2] = W[l][n, k0 + kk]
            off += N * 2 * w
    pos = boff
    assert boff % 1024 == 0
    for l in range(len(dims) - 1):
        ew[pos // 2: pos // 2 + dims[l + 1]] = b[l]
        pos += 2 * dims[l + 1]
    assert pos == size
    assert np.array_equal(words, ew)


def test_pack_is_a_permutation(orc):
    dims = (48, 64, 112, 16)
    rng = np.random.default_rng(3)
    total = sum(dims[l] * dims[l + 1] + dims[l + 1] for l in range(len(dims) - 1))
    vals = rng.permutation(np.arange(1, total + 1)).astype(np.uint16)
    W, b, p = [], [], 0
    for l in range(len(dims) - 1):
        K, N = dims[l], dims[l + 1]
        W.append(vals[p:p + N * K].reshape(N, K)); p += N * K
        b.append(vals[p:p + N]); p += N
    blob = orc.pack(dims, W, b).view(np.uint16)
    nz = blob[blob != 0]
    assert nz.size == total
    assert np.array_equal(np.sort(nz), np.arange(1, total + 1, dtype=np.uint16))


def test_packed_sizes(orc):
    # tiny: 7 images of 32x32 (2048 B each, one 64-byte-swizzle segment) and a
    # 16x32 image (1024 B), then 7*32+16 = 240 biases (480 B).
    assert orc.packed_layout(synth.WORKLOADS["tiny"].dims) == (
        7 * 2048 + 1024 + 480, [i * 2048 for i in range(8)], 7 * 2048 + 1024)
    # page: 48 -> 64 image = segment 64x(32 wide) 4096 B + segment 64x(16 wide)
    # 2048 B; six 64x64 images of 8192 B; 16x64 image 2048 B; 464 biases.
    size, img, boff = orc.packed_layout(synth.WORKLOADS["page"].dims)
    assert img == [0, 6144] + [6144 + 8192 * i for i in range(1, 7)]
    assert boff == 6144 + 6 * 8192 + 2048
    assert size == boff + 2 * (7 * 64 + 16)
    # hetero: weights 168,960 elements, no padding needed anywhere
    size, img, boff = orc.packed_layout(synth.WORKLOADS["hetero"].dims)
    assert boff == 2 * 168960 and size == boff + 2 * 1040


@pytest.mark.parametrize("dims", [(8, 16), (32, 24), (272, 16), (32,) * 18])
def test_packed_layout_rejects(orc, dims):
    with pytest.raises(ValueError):
        orc.packed_layout(dims)
