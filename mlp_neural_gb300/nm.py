"""Thin ctypes binding of libnmmlp (include/nm_mlp.h): same names, argument
marshalling only. Every step of inference runs in the library's CUDA
kernels; there is no other implementation behind these calls, and a missing
library raises instead of falling back.

Tensors are PyTorch CUDA tensors (used for device memory and streams only);
raw device addresses (ints) are accepted wherever a tensor is.
"""
from __future__ import annotations

import ctypes
import os
import threading

NM_OK = 0
NM_ERR_INVALID_ARG = 1
NM_ERR_UNSUPPORTED = 2
NM_ERR_NOT_PACKED = 3
NM_ERR_OOM = 4
NM_ERR_CUDA = 5
NM_ERR_TIMEOUT = 6
NM_ERR_RANGE_CHECK = 7

NM_VARIANT_FUSED = 0
NM_VARIANT_ROWMAJOR_WEIGHTS = 1
NM_VARIANT_SCALAR_ACTIVATION = 2
NM_VARIANT_PAIRED_TILES = 3
NM_VARIANT_FP8_WEIGHTS = 4

# NM_CHECKED=1 in the environment selects the checking build
# (libnmmlp_check.so, kernels compiled with NM_RANGE_CHECKS).
_PKG = os.path.dirname(os.path.abspath(__file__))
CHECKED = os.environ.get("NM_CHECKED", "") == "1"
LIB_PATH = os.path.join(_PKG, "libnmmlp_check.so" if CHECKED else "libnmmlp.so")

# Every symbol include/nm_mlp.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
SIGNATURES = {
    "nm_abi_version": (ctypes.c_int32, []),
    "nm_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "nm_mlp_create": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(_P)]),
    "nm_mlp_packed_size": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_size_t)]),
    "nm_mlp_pack_weights": (ctypes.c_int, [_P, _P, _P, _P]),
    "nm_mlp_unpack_weights": (ctypes.c_int, [_P, _P, _P, _P]),
    "nm_mlp_packed_blob": (ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    "nm_mlp_packed_fp8": (ctypes.c_int, [_P, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    "nm_mlp_infer": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P, _P]),
    "nm_mlp_infer_host": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P, _P]),
    "nm_mlp_set_host_chunk": (ctypes.c_int, [_P, ctypes.c_int64]),
    "nm_mlp_set_variant": (ctypes.c_int, [_P, ctypes.c_int]),
    "nm_mlp_device_status": (ctypes.c_int, [_P, _P]),
    "nm_mlp_set_wait_limit": (ctypes.c_int, [_P, ctypes.c_uint64]),
    "nm_mlp_set_test_stall": (ctypes.c_int, [_P, ctypes.c_int32]),
    "nm_checking_build": (ctypes.c_int32, []),
    "nm_mlp_set_test_check_limit": (ctypes.c_int, [_P, ctypes.c_uint32]),
    "nm_mlp_infer_noalloc": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P, _P, ctypes.c_int64, _P, _P]),
    "nm_mlp_plan": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int, ctypes.c_uint32, _P]),
    "nm_mlp_destroy": (None, [_P]),
}

_lock = threading.Lock()
_lib = None


class NmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


def lib():
    """Open libnmmlp.so, or libnmmlp_check.so under NM_CHECKED=1 (both built
    by __graft_entry__.build(); ``python -m mlp_neural_gb300.build [--checked]``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m mlp_neural_gb300.build"
                    + (" --checked" if CHECKED else "") + "` (there is no fallback path)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def status_str(status: int) -> str:
    return lib().nm_status_str(int(status)).decode()


def _check(status: int, what: str):
    if status != NM_OK:
        raise NmError(status, what)


def _addr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


class Plan(ctypes.Structure):
    """nm_plan: how the fused kernel runs a network (see nm_mlp_plan)."""
    _fields_ = [("tile_slots", ctypes.c_int32), ("warps_per_slot", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("streamed_weights", ctypes.c_int32),
                ("weight_stages", ctypes.c_int32), ("input_stages", ctypes.c_int32),
                ("output_buffers", ctypes.c_int32), ("smem_bytes", ctypes.c_uint32),
                ("tmem_columns", ctypes.c_uint32), ("issuing_warps", ctypes.c_int32),
                ("a_tmem_k", ctypes.c_int32)]


GB300_SMEM_OPTIN = 232448  # opt-in shared memory per block on GB300, bytes


def plan(dims, variant: int = NM_VARIANT_FUSED, smem_optin: int = GB300_SMEM_OPTIN) -> dict:
    """nm_mlp_plan: the kernel's plan for a network, computed on the host
    (no device needed). Raises NmError if no plan fits."""
    d = (ctypes.c_int32 * len(dims))(*[int(v) for v in dims])
    p = Plan()
    _check(lib().nm_mlp_plan(d, len(dims), int(variant), int(smem_optin), ctypes.byref(p)),
           "nm_mlp_plan")
    return {name: getattr(p, name) for name, _ in Plan._fields_}


def infer_noalloc(dims, W, b, x, out, stream=None) -> int:
    """nm_mlp_infer_noalloc: inference without any device allocation by the
    library (for callers that cannot allocate); returns the status code."""
    d = (ctypes.c_int32 * len(dims))(*[int(v) for v in dims])
    Wp = (ctypes.c_void_p * len(W))(*[_addr(w) for w in W])
    bp = (ctypes.c_void_p * len(b))(*[_addr(v) for v in b])
    n = x.shape[0] if hasattr(x, "shape") else 0
    return lib().nm_mlp_infer_noalloc(d, len(dims), Wp, bp, _addr(x), int(n), _addr(out),
                                      _stream(stream))


class MLP:
    """Owns one nm_mlp handle (dims, packed weights on the device)."""

    def __init__(self, dims):
        self.dims = [int(d) for d in dims]
        arr = (ctypes.c_int32 * len(self.dims))(*self.dims)
        h = ctypes.c_void_p()
        _check(lib().nm_mlp_create(arr, len(self.dims), ctypes.byref(h)), "nm_mlp_create")
        self._h = h

    @property
    def handle(self) -> int:
        return self._h.value

    @property
    def n_layers(self) -> int:
        return len(self.dims) - 1

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().nm_mlp_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def packed_size(self) -> int:
        n = ctypes.c_size_t()
        _check(lib().nm_mlp_packed_size(self._h, ctypes.byref(n)), "nm_mlp_packed_size")
        return n.value

    def packed_blob(self) -> int:
        p = ctypes.c_void_p()
        _check(lib().nm_mlp_packed_blob(self._h, ctypes.byref(p)), "nm_mlp_packed_blob")
        return p.value

    def packed_fp8(self):
        """(device address, bytes) of the E4M3 weight images."""
        p = _P()
        n = ctypes.c_size_t()
        _check(lib().nm_mlp_packed_fp8(self._h, ctypes.byref(p), ctypes.byref(n)), "nm_mlp_packed_fp8")
        return int(p.value or 0), int(n.value)

    def pack_weights(self, W, b, stream=None):
        Wp = (ctypes.c_void_p * len(W))(*[_addr(w) for w in W])
        bp = (ctypes.c_void_p * len(b))(*[_addr(v) for v in b])
        _check(lib().nm_mlp_pack_weights(self._h, Wp, bp, _stream(stream)), "nm_mlp_pack_weights")

    def unpack_weights(self, W, b, stream=None):
        Wp = (ctypes.c_void_p * len(W))(*[_addr(w) for w in W])
        bp = (ctypes.c_void_p * len(b))(*[_addr(v) for v in b])
        _check(lib().nm_mlp_unpack_weights(self._h, Wp, bp, _stream(stream)),
               "nm_mlp_unpack_weights")

    def infer_raw(self, in_ptr: int, n: int, out_ptr: int, stream=None) -> int:
        """nm_mlp_infer on raw addresses; returns the status code."""
        return lib().nm_mlp_infer(self._h, in_ptr, int(n), out_ptr, _stream(stream))

    def infer(self, x, out=None, stream=None):
        """out[n, d_L] = network(x[n, d_0]); both FP16 CUDA tensors."""
        import torch
        n = x.shape[0]
        if out is None:
            out = torch.empty((n, self.dims[-1]), dtype=torch.float16, device=x.device)
        _check(self.infer_raw(_addr(x), n, _addr(out), stream), "nm_mlp_infer")
        return out

    def infer_host_raw(self, in_ptr: int, n: int, out_ptr: int, stream=None) -> int:
        """nm_mlp_infer_host on raw host addresses; returns the status code."""
        return lib().nm_mlp_infer_host(self._h, in_ptr, int(n), out_ptr, _stream(stream))

    def infer_host(self, x, out=None, stream=None):
        """out[n, d_L] = network(x[n, d_0]) with both FP16 tensors in host
        memory (page-locked for overlapped copies). Asynchronous on `stream`:
        synchronise it before reading `out`."""
        import torch
        if x.device.type != "cpu" or x.dtype != torch.float16 or not x.is_contiguous():
            raise ValueError("infer_host wants a contiguous FP16 host tensor")
        n = x.shape[0]
        if out is None:
            out = torch.empty((n, self.dims[-1]), dtype=torch.float16, pin_memory=True)
        if out.device.type != "cpu" or out.dtype != torch.float16 or not out.is_contiguous():
            raise ValueError("infer_host writes a contiguous FP16 host tensor")
        _check(self.infer_host_raw(x.data_ptr(), n, out.data_ptr(), stream), "nm_mlp_infer_host")
        return out

    def set_host_chunk(self, rows: int):
        _check(lib().nm_mlp_set_host_chunk(self._h, int(rows)), "nm_mlp_set_host_chunk")

    def set_variant(self, v: int):
        _check(lib().nm_mlp_set_variant(self._h, int(v)), "nm_mlp_set_variant")

    def device_status(self, stream=None) -> int:
        return lib().nm_mlp_device_status(self._h, _stream(stream))

    def set_wait_limit(self, ns: int):
        _check(lib().nm_mlp_set_wait_limit(self._h, int(ns)), "nm_mlp_set_wait_limit")

    def set_test_stall(self, enable: bool):
        _check(lib().nm_mlp_set_test_stall(self._h, 1 if enable else 0), "nm_mlp_set_test_stall")

    def set_test_check_limit(self, tmem_columns: int):
        _check(lib().nm_mlp_set_test_check_limit(self._h, int(tmem_columns)),
               "nm_mlp_set_test_check_limit")


def checking_build() -> bool:
    """nm_checking_build: True for the library compiled with NM_RANGE_CHECKS."""
    return bool(lib().nm_checking_build())
