"""The C ABI from a C program on the GPU: a C99 client (gcc, CUDA runtime for
its own buffers) creates a handle, packs row-major weights, and runs the
page-shaped network through nm_mlp_infer (device buffers), nm_mlp_infer_host
(pinned host buffers) and nm_mlp_infer_noalloc. The three outputs must be
bit-identical and match the oracle; no Python binding is involved in the
calls."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from mlp_neural_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

C_CLIENT = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "nm_mlp.h"

#define CK(x) do { if ((x) != 0) { fprintf(stderr, "fail %s:%d\n", __FILE__, __LINE__); return 1; } } while (0)

static void *read_file(const char *path, size_t bytes) {
    FILE *f = fopen(path, "rb");
    void *p = malloc(bytes);
    if (!f || !p || fread(p, 1, bytes, f) != bytes) { fprintf(stderr, "read %s\n", path); exit(2); }
    fclose(f);
    return p;
}

int main(int argc, char **argv) {
    /* argv: dir, n, d_0 .. d_L */
    const char *dir = argv[1];
    const int64_t n = atoll(argv[2]);
    const int32_t n_dims = argc - 3, L = n_dims - 1;
    int32_t dims[32];
    void *W[16], *b[16];
    char path[4096];
    int l;
    nm_mlp *h = NULL;
    uint16_t *x, *y_dev, *y_host, *y_noalloc;
    void *dx, *dy, *px, *py;
    size_t out_bytes;
    FILE *f;
    for (l = 0; l < n_dims; ++l) dims[l] = atoi(argv[3 + l]);
    for (l = 0; l < L; ++l) {
        const size_t wb = (size_t)dims[l] * dims[l + 1] * 2, bb = (size_t)dims[l + 1] * 2;
        void *hw, *hb;
        snprintf(path, sizeof path, "%s/W%d.bin", dir, l);
        hw = read_file(path, wb);
        snprintf(path, sizeof path, "%s/b%d.bin", dir, l);
        hb = read_file(path, bb);
        CK(cudaMalloc(&W[l], wb));
        CK(cudaMalloc(&b[l], bb));
        CK(cudaMemcpy(W[l], hw, wb, cudaMemcpyHostToDevice));
        CK(cudaMemcpy(b[l], hb, bb, cudaMemcpyHostToDevice));
        free(hw);
        free(hb);
    }
    snprintf(path, sizeof path, "%s/x.bin", dir);
    x = (uint16_t *)read_file(path, (size_t)n * dims[0] * 2);
    out_bytes = (size_t)n * dims[L] * 2;
    y_dev = (uint16_t *)malloc(out_bytes);
    y_noalloc = (uint16_t *)malloc(out_bytes);

    CK(nm_mlp_create(dims, n_dims, &h));
    CK(nm_mlp_pack_weights(h, (const void *const *)W, (const void *const *)b, NULL));

    /* device buffers */
    CK(cudaMalloc(&dx, (size_t)n * dims[0] * 2));
    CK(cudaMalloc(&dy, out_bytes));
    CK(cudaMemcpy(dx, x, (size_t)n * dims[0] * 2, cudaMemcpyHostToDevice));
    CK(nm_mlp_infer(h, dx, n, dy, NULL));
    CK(nm_mlp_device_status(h, NULL));
    CK(cudaMemcpy(y_dev, dy, out_bytes, cudaMemcpyDeviceToHost));

    /* pinned host buffers */
    CK(cudaMallocHost(&px, (size_t)n * dims[0] * 2));
    CK(cudaMallocHost(&py, out_bytes));
    memcpy(px, x, (size_t)n * dims[0] * 2);
    CK(nm_mlp_set_host_chunk(h, 1024));
    CK(nm_mlp_infer_host(h, px, n, py, NULL));
    CK(cudaDeviceSynchronize());
    CK(nm_mlp_device_status(h, NULL));
    y_host = (uint16_t *)py;

    /* no allocation by the library */
    CK(cudaMemset(dy, 0, out_bytes));
    CK(nm_mlp_infer_noalloc(dims, n_dims, (const void *const *)W, (const void *const *)b, dx, n, dy, NULL));
    CK(cudaMemcpy(y_noalloc, dy, out_bytes, cudaMemcpyDeviceToHost));

    snprintf(path, sizeof path, "%s/y.bin", dir);
    f = fopen(path, "wb");
    if (!f) return 3;
    fwrite(y_dev, 1, out_bytes, f);
    fwrite(y_host, 1, out_bytes, f);
    fwrite(y_noalloc, 1, out_bytes, f);
    fclose(f);

    nm_mlp_destroy(h);
    CK(cudaFreeHost(px));
    CK(cudaFreeHost(py));
    CK(cudaFree(dx));
    CK(cudaFree(dy));
    for (l = 0; l < L; ++l) { CK(cudaFree(W[l])); CK(cudaFree(b[l])); }
    free(x);
    free(y_dev);
    free(y_noalloc);
    printf("ok\n");
    return 0;
}
"""


def test_c_client_three_entry_points(orc, tmp_path):
    from gpu_util import assert_close, nm
    lib = nm()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib.LIB_PATH)
    name = os.path.basename(lib.LIB_PATH)[3:-3]
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                        str(src), "-o", str(exe), "-L", libdir, f"-l{name}",
                        "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                        f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    dims = synth.WORKLOADS["page"].dims
    n = 152 * 128 + 77
    W, b, x = synth.small_net_inputs(dims, seed=91, n=n)
    for l in range(len(dims) - 1):
        W[l].astype(np.uint16).tofile(tmp_path / f"W{l}.bin")
        b[l].astype(np.uint16).tofile(tmp_path / f"b{l}.bin")
    x.astype(np.uint16).tofile(tmp_path / "x.bin")
    r = subprocess.run([str(exe), str(tmp_path), str(n)] + [str(d) for d in dims],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
    y = np.fromfile(tmp_path / "y.bin", dtype=np.uint16).reshape(3, n, dims[-1])
    assert np.array_equal(y[0], y[1]), "nm_mlp_infer_host differs from nm_mlp_infer"
    assert np.array_equal(y[0], y[2]), "nm_mlp_infer_noalloc differs from nm_mlp_infer"
    assert_close(y[0], orc.forward(dims, W, b, x), "C client")
