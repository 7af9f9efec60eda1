"""CPU oracle for the fused FP16 MLP (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` import this package. The product library never does, and this
package imports nothing from ``mlp_neural_gb300`` except that both sides take
their seeded inputs from ``mlp_neural_gb300.synth``, which holds none of the
method's arithmetic.

The arithmetic lives in ``nm_oracle.c`` (plain C, single-threaded); this file
only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MAX_LAYERS = 16


def build(force: bool = False) -> str:
    """Compile nm_oracle.c into oracle/liboracle.so with gcc.

    -ffp-contract=off keeps every FP32 multiply and add separate, as written.
    (The products are exact in FP32 anyway, so a fused multiply-add would
    round identically; the flag keeps the source and the binary saying the
    same thing.)
    """
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u16, f32 = ctypes.c_uint16, ctypes.c_float
            P = ctypes.c_void_p
            L.or_f16_to_f32.argtypes = [u16]
            L.or_f16_to_f32.restype = f32
            L.or_f32_to_f16.argtypes = [f32]
            L.or_f32_to_f16.restype = u16
            L.or_slope_f16.argtypes = []
            L.or_slope_f16.restype = u16
            L.or_leaky_max.argtypes = [u16]
            L.or_leaky_max.restype = u16
            L.or_leaky_branchy.argtypes = [u16]
            L.or_leaky_branchy.restype = u16
            L.or_mlp_forward.argtypes = [P, ctypes.c_int32, P, P, P, ctypes.c_int64, P]
            L.or_mlp_forward.restype = ctypes.c_int
            L.or_packed_layout.argtypes = [P, ctypes.c_int32, P, P]
            L.or_packed_layout.restype = ctypes.c_int64
            L.or_pack.argtypes = [P, ctypes.c_int32, P, P, P]
            L.or_pack.restype = ctypes.c_int
            L.or_unpack.argtypes = [P, ctypes.c_int32, P, P, P]
            L.or_unpack.restype = ctypes.c_int
            L.or_mlp_forward_fp8.argtypes = [P, ctypes.c_int32, P, P, P, ctypes.c_int64, P]
            L.or_mlp_forward_fp8.restype = ctypes.c_int
            L.or_fp8_layout.argtypes = [P, ctypes.c_int32, P]
            L.or_fp8_layout.restype = ctypes.c_int64
            L.or_pack_fp8.argtypes = [P, ctypes.c_int32, P, P]
            L.or_pack_fp8.restype = ctypes.c_int
            L.or_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            L.or_e4m3_to_f32.restype = f32
            L.or_f16_to_e4m3.argtypes = [u16]
            L.or_f16_to_e4m3.restype = ctypes.c_uint8
            for name in ("or_f16_to_f32_n", "or_f32_to_f16_n", "or_leaky_max_n",
                         "or_leaky_branchy_n", "or_e4m3_to_f32_n", "or_f16_to_e4m3_n"):
                getattr(L, name).argtypes = [P, ctypes.c_int64, P]
                getattr(L, name).restype = None
            _lib = L
        return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def _dims_arr(dims):
    return np.ascontiguousarray(np.asarray(dims, dtype=np.int32))


def f16_to_f32(h: int) -> float:
    return lib().or_f16_to_f32(int(h))


def f32_to_f16(x: float) -> int:
    return lib().or_f32_to_f16(float(x))


def slope_f16() -> int:
    return lib().or_slope_f16()


def leaky_max(h: int) -> int:
    return lib().or_leaky_max(int(h))


def leaky_branchy(h: int) -> int:
    return lib().or_leaky_branchy(int(h))


def f16_to_f32_array(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().or_f16_to_f32_n(_ptr(h), h.size, _ptr(out))
    return out


def f32_to_f16_array(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().or_f32_to_f16_n(_ptr(x), x.size, _ptr(out))
    return out


def leaky_max_array(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.uint16)
    lib().or_leaky_max_n(_ptr(h), h.size, _ptr(out))
    return out


def leaky_branchy_array(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.uint16)
    lib().or_leaky_branchy_n(_ptr(h), h.size, _ptr(out))
    return out


def e4m3_to_f32_array(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float32)
    lib().or_e4m3_to_f32_n(_ptr(c), c.size, _ptr(out))
    return out


def f16_to_e4m3_array(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.uint8)
    lib().or_f16_to_e4m3_n(_ptr(h), h.size, _ptr(out))
    return out


def forward(dims, W, b, x) -> np.ndarray:
    """Evaluate the network on every row of ``x``.

    ``dims`` = [d_0, ..., d_L]; ``W[l]`` is an FP16-bits (uint16) array of
    shape [d_{l+1}, d_l]; ``b[l]`` has d_{l+1} entries; ``x`` is uint16
    [n, d_0]. Returns uint16 [n, d_L].
    """
    return _forward(lib().or_mlp_forward, dims, W, b, x)


def forward_fp8(dims, W, b, x) -> np.ndarray:
    """The narrow-precision pass (E4M3 weights of layers 2..L and E4M3
    activations feeding them), same arguments as ``forward``."""
    return _forward(lib().or_mlp_forward_fp8, dims, W, b, x)


def _forward(fn, dims, W, b, x) -> np.ndarray:
    dims = _dims_arr(dims)
    L = len(dims) - 1
    W = [np.ascontiguousarray(w, dtype=np.uint16) for w in W]
    b = [np.ascontiguousarray(v, dtype=np.uint16) for v in b]
    assert len(W) == L and len(b) == L
    for l in range(L):
        assert W[l].shape == (dims[l + 1], dims[l]), (l, W[l].shape)
        assert b[l].shape == (dims[l + 1],)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert x.ndim == 2 and x.shape[1] == dims[0]
    y = np.zeros((x.shape[0], dims[-1]), dtype=np.uint16)
    rc = fn(_ptr(dims), L, _ptr_array(W), _ptr_array(b), _ptr(x), x.shape[0], _ptr(y))
    if rc != 0:
        raise ValueError(f"the oracle rejected dims {dims.tolist()} (rc={rc})")
    return y


def packed_layout(dims):
    """(blob_size, [image offsets], bias offset) of the packed blob."""
    dims = _dims_arr(dims)
    L = len(dims) - 1
    img = np.zeros(MAX_LAYERS, dtype=np.int64)
    boff = np.zeros(1, dtype=np.int64)
    size = lib().or_packed_layout(_ptr(dims), L, _ptr(img), _ptr(boff))
    if size < 0:
        raise ValueError(f"unsupported dims {dims.tolist()}")
    return int(size), [int(v) for v in img[:L]], int(boff[0])


def pack(dims, W, b) -> np.ndarray:
    dims = _dims_arr(dims)
    L = len(dims) - 1
    size, _, _ = packed_layout(dims)
    W = [np.ascontiguousarray(w, dtype=np.uint16) for w in W]
    b = [np.ascontiguousarray(v, dtype=np.uint16) for v in b]
    blob = np.zeros(size, dtype=np.uint8)
    rc = lib().or_pack(_ptr(dims), L, _ptr_array(W), _ptr_array(b), _ptr(blob))
    if rc != 0:
        raise ValueError("or_pack failed")
    return blob


def unpack(dims, blob):
    dims = _dims_arr(dims)
    L = len(dims) - 1
    W = [np.zeros((dims[l + 1], dims[l]), dtype=np.uint16) for l in range(L)]
    b = [np.zeros(dims[l + 1], dtype=np.uint16) for l in range(L)]
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    rc = lib().or_unpack(_ptr(dims), L, _ptr(blob), _ptr_array(W), _ptr_array(b))
    if rc != 0:
        raise ValueError("or_unpack failed")
    return W, b


def fp8_layout(dims):
    """(region size, [image offsets, None for layer 0]) of the E4M3 images."""
    dims = _dims_arr(dims)
    L = len(dims) - 1
    img = np.zeros(MAX_LAYERS, dtype=np.int64)
    size = lib().or_fp8_layout(_ptr(dims), L, _ptr(img))
    if size < 0:
        raise ValueError(f"no E4M3 images for dims {dims.tolist()}")
    return int(size), [None] + [int(v) for v in img[1:L]]


def pack_fp8(dims, W) -> np.ndarray:
    dims = _dims_arr(dims)
    L = len(dims) - 1
    size, _ = fp8_layout(dims)
    W = [np.ascontiguousarray(w, dtype=np.uint16) for w in W]
    region = np.zeros(size, dtype=np.uint8)
    rc = lib().or_pack_fp8(_ptr(dims), L, _ptr_array(W), _ptr(region))
    if rc != 0:
        raise ValueError("or_pack_fp8 failed")
    return region
