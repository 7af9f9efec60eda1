"""Helpers for the GPU tests: build/load the library, move uint16 FP16 bits
between numpy and torch CUDA tensors, read raw device memory, run the oracle.
"""
import ctypes
import glob
import os

import numpy as np

TOL_ABS = 1e-2
TOL_REL = 1e-2


def nm():
    """The binding, its library built first (the checking build when the
    process runs with NM_CHECKED=1)."""
    from mlp_neural_gb300 import build, nm as _nm
    build.build(checked=_nm.CHECKED)
    return _nm


def to_dev(a16: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a16).view(np.int16)).cuda().view(torch.float16)


def to_host(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


_cudart = None


def _rt():
    global _cudart
    if _cudart is None:
        import torch
        cands = glob.glob(os.path.join(os.path.dirname(torch.__file__), "..", "nvidia", "*", "lib",
                                       "libcudart.so*"))
        cands += ["libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"]
        for c in cands:
            try:
                _cudart = ctypes.CDLL(c)
                break
            except OSError:
                continue
        _cudart.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    return _cudart


def read_device(ptr: int, nbytes: int) -> np.ndarray:
    import torch
    torch.cuda.synchronize()
    out = np.empty(nbytes, np.uint8)
    rc = _rt().cudaMemcpy(out.ctypes.data, ptr, nbytes, 2)  # cudaMemcpyDeviceToHost
    assert rc == 0, rc
    return out


def make_net(dims, W, b):
    """Create a library handle and pack W/b (uint16 numpy) into it."""
    lib = nm()
    m = lib.MLP(dims)
    Wd = [to_dev(w) for w in W]
    bd = [to_dev(v) for v in b]
    m.pack_weights(Wd, bd)
    import torch
    torch.cuda.synchronize()
    return m


def assert_close(gpu16: np.ndarray, cpu16: np.ndarray, what=""):
    g = gpu16.view(np.float16).astype(np.float64)
    c = cpu16.view(np.float16).astype(np.float64)
    assert g.shape == c.shape, (g.shape, c.shape)
    err = np.abs(g - c)
    bound = TOL_ABS + TOL_REL * np.abs(c)
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, (f"{what}: {len(bad)} elements outside |gpu-cpu| <= 1e-2 + 1e-2|cpu|; "
                           f"first {bad[:5].tolist()} gpu={g[tuple(bad[0])]} cpu={c[tuple(bad[0])]}")
    return float(err.max()) if err.size else 0.0


def fp8_rows_parallel(orc, dims, W, b, x, y_gpu, row_frac, tol_abs, tol_rel, chunk=32768,
                      threads=None):
    """Every row of y_gpu against the oracle's E4M3 pass on all host cores
    (as check_rows_parallel): at most row_frac of the rows may differ at all,
    and no element by more than tol_abs + tol_rel |cpu|. Returns (rows
    checked, rows that differ, largest |gpu - cpu|, threads used)."""
    from concurrent.futures import ThreadPoolExecutor
    n = x.shape[0]
    assert y_gpu.shape == (n, dims[-1])
    if threads is None:
        threads = os.cpu_count() or 1

    def work(r0):
        r1 = min(n, r0 + chunk)
        ref = orc.forward_fp8(dims, W, b, x[r0:r1]).view(np.float16).astype(np.float64)
        got = y_gpu[r0:r1].view(np.float16).astype(np.float64)
        err = np.abs(got - ref)
        badm = ~(err <= tol_abs + tol_rel * np.abs(ref))
        first = None
        if badm.any():
            i, j = np.argwhere(badm)[0]
            first = (r0 + int(i), int(j), float(got[i, j]), float(ref[i, j]))
        return (int((err.max(axis=1) > 0).sum()), int(badm.sum()),
                float(np.nanmax(err)) if err.size else 0.0, first)

    with ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(work, range(0, n, chunk)))
    rows = sum(r[0] for r in res)
    bad = sum(r[1] for r in res)
    firsts = [r[3] for r in res if r[3] is not None]
    assert bad == 0, (f"{bad} elements outside |gpu-cpu| <= {tol_abs} + {tol_rel}|cpu|; "
                      f"first (row, col, gpu, cpu) = {firsts[0]}")
    assert rows <= row_frac * n, f"{rows} of {n} rows differ from the oracle"
    return n, rows, max(r[2] for r in res), threads


def check_rows_parallel(orc, dims, W, b, x, y_gpu, chunk=32768, threads=None):
    """Every row of y_gpu (uint16 FP16 bits, [n, d_L]) against the oracle on
    the same inputs, within |gpu - cpu| <= 1e-2 + 1e-2|cpu| per element.

    The oracle stays single-threaded per call; contiguous row ranges run on a
    thread pool over all host cores (ctypes releases the GIL during the call),
    and each worker compares its own range, so memory stays bounded. Returns
    (rows checked, largest |gpu - cpu|, threads used)."""
    from concurrent.futures import ThreadPoolExecutor
    n = x.shape[0]
    assert y_gpu.shape == (n, dims[-1])
    if threads is None:
        threads = os.cpu_count() or 1

    def work(r0):
        r1 = min(n, r0 + chunk)
        ref = orc.forward(dims, W, b, x[r0:r1]).view(np.float16).astype(np.float64)
        got = y_gpu[r0:r1].view(np.float16).astype(np.float64)
        err = np.abs(got - ref)
        bad = ~(err <= TOL_ABS + TOL_REL * np.abs(ref))
        first = None
        if bad.any():
            i, j = np.argwhere(bad)[0]
            first = (r0 + int(i), int(j), float(got[i, j]), float(ref[i, j]))
        return int(bad.sum()), first, float(err.max()) if err.size else 0.0

    with ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(work, range(0, n, chunk)))
    n_bad = sum(r[0] for r in res)
    firsts = [r[1] for r in res if r[1] is not None]
    assert n_bad == 0, (f"{n_bad} elements outside |gpu-cpu| <= 1e-2 + 1e-2|cpu|; "
                        f"first (row, col, gpu, cpu) = {firsts[0]}")
    return n, max(r[2] for r in res), threads
