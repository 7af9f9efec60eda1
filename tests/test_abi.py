"""The C-ABI library loads on a machine without a GPU and exports every symbol
include/nm_mlp.h declares; host-side argument checks answer without touching
a device. (CPU only: no compute call is made.)"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nm_mlp.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nm_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def nmlib():
    from mlp_neural_gb300 import build, nm
    build.build(checked=nm.CHECKED)
    return nm


def test_header_declares_the_problem_statement_calls():
    names = _declared_functions()
    for required in ("nm_mlp_create", "nm_mlp_pack_weights", "nm_mlp_infer", "nm_mlp_destroy",
                     "nm_mlp_packed_size"):
        assert required in names


def test_library_exports_every_declared_symbol(nmlib):
    L = ctypes.CDLL(nmlib.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    # the binding covers exactly the declared calls
    assert sorted(nmlib.SIGNATURES) == _declared_functions()


def test_checking_build_exports_every_declared_symbol(nmlib):
    """libnmmlp_check.so (NM_RANGE_CHECKS) builds, loads without a GPU,
    exports the same calls and says which build it is."""
    from mlp_neural_gb300 import build
    path = build.build(checked=True)
    L = ctypes.CDLL(path)
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    L.nm_checking_build.restype = ctypes.c_int32
    assert L.nm_checking_build() == 1
    normal = ctypes.CDLL(build.build())
    normal.nm_checking_build.restype = ctypes.c_int32
    assert normal.nm_checking_build() == 0
    L.nm_mlp_set_test_check_limit.argtypes = [ctypes.c_void_p, ctypes.c_uint32]
    assert L.nm_mlp_set_test_check_limit(None, 16) == nmlib.NM_ERR_INVALID_ARG
    L.nm_status_str.restype = ctypes.c_char_p
    assert L.nm_status_str(nmlib.NM_ERR_RANGE_CHECK) == b"NM_ERR_RANGE_CHECK"


def test_status_strings(nmlib):
    for code in range(8):
        assert nmlib.status_str(code).startswith("NM_")
    assert nmlib.status_str(nmlib.NM_ERR_TIMEOUT) == "NM_ERR_TIMEOUT"
    assert nmlib.lib().nm_abi_version() == 4


@pytest.mark.parametrize("dims,expect", [
    ((32,), 1),                 # fewer than two widths
    ((32, 24), 2),              # not a multiple of 16
    ((32, 272), 2),             # wider than 256
    ((16,) * 18, 2),            # more than 16 layers
])
def test_create_rejects_bad_dims_on_the_host(nmlib, dims, expect):
    h = ctypes.c_void_p()
    arr = (ctypes.c_int32 * len(dims))(*dims)
    assert nmlib.lib().nm_mlp_create(arr, len(dims), ctypes.byref(h)) == expect
    assert h.value is None


def test_null_handles_are_invalid(nmlib):
    L = nmlib.lib()
    assert L.nm_mlp_infer(None, None, 0, None, None) == nmlib.NM_ERR_INVALID_ARG
    assert L.nm_mlp_set_variant(None, 0) == nmlib.NM_ERR_INVALID_ARG
    assert L.nm_mlp_device_status(None, None) == nmlib.NM_ERR_INVALID_ARG
    n = ctypes.c_size_t()
    assert L.nm_mlp_packed_size(None, ctypes.byref(n)) == nmlib.NM_ERR_INVALID_ARG
    L.nm_mlp_destroy(None)  # no-op


def test_noalloc_argument_checks_on_the_host(nmlib):
    L = nmlib.lib()
    dims = (ctypes.c_int32 * 2)(32, 24)
    null2 = (ctypes.c_void_p * 1)(None)
    assert L.nm_mlp_infer_noalloc(dims, 2, null2, null2, None, 4, None, None) == nmlib.NM_ERR_UNSUPPORTED
    dims = (ctypes.c_int32 * 2)(32, 16)
    assert L.nm_mlp_infer_noalloc(dims, 2, null2, null2, None, 4, None, None) == nmlib.NM_ERR_INVALID_ARG


def test_host_path_argument_checks_on_the_host(nmlib):
    L = nmlib.lib()
    assert L.nm_mlp_infer_host(None, None, 4, None, None) == nmlib.NM_ERR_INVALID_ARG
    assert L.nm_mlp_set_host_chunk(None, 0) == nmlib.NM_ERR_INVALID_ARG


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "nm_mlp.h"

int main(void) {
    const int32_t page[9] = {48, 64, 64, 64, 64, 64, 64, 64, 16};
    const int32_t bad[2] = {32, 24};
    nm_plan plan;
    nm_mlp *h = (nm_mlp *)1;
    nm_status st;
    printf("abi %d\n", (int)nm_abi_version());
    printf("str %s\n", nm_status_str(NM_ERR_RANGE_CHECK));
    st = nm_mlp_create(bad, 2, &h);
    printf("create_bad %d %d\n", (int)st, h == NULL);
    memset(&plan, 0, sizeof(plan));
    st = nm_mlp_plan(page, 9, NM_VARIANT_FUSED, 232448u, &plan);
    printf("plan %d %d %d %d %u\n", (int)st, (int)plan.tile_slots, (int)plan.threads,
           (int)plan.streamed_weights, (unsigned)plan.tmem_columns);
    printf("checking %d\n", (int)nm_checking_build());
    nm_mlp_destroy(NULL);
    return 0;
}
"""


def test_header_is_plain_c_and_links(nmlib, tmp_path):
    """A C99 program (gcc, -Wall -Werror -pedantic) includes the header, links
    against the library and makes the calls that need no device: the boundary
    holds for C callers, not only for the Python binding."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(nmlib.LIB_PATH)
    lib = os.path.basename(nmlib.LIB_PATH)[3:-3]
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, f"-l{lib}", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert out["abi"] == "4"
    assert out["str"] == "NM_ERR_RANGE_CHECK"
    assert out["create_bad"] == "2 1"
    assert out["plan"] == "0 5 896 0 512"
    assert out["checking"] == ("1" if nmlib.CHECKED else "0")
