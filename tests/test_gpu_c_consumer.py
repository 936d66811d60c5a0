"""A plain C11 program drives the library on the GPU through the CUDA runtime
alone (cudaMalloc, cudaMemcpy, a stream): the fused paged slot map + write of
a small batch, then the gather of each request's span.  It prints what it
read back; the test compares that with the oracle on the same inputs."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_39_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

pytestmark = pytest.mark.gpu

T, B, H, D, STRIDE = 16, 64, 2, 8, 4
QSL = [0, 3, 4, 6]
POS = [0, 1, 17, 40, 5, 63]
TABLE = [[5, 9, 0, 0], [7, 11, 13, 2], [0, 0, 0, 0]]
G0 = [0, 30, 60]
G1 = [18, 41, 64]

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include <cuda_runtime_api.h>
#include "kvpaged.h"

enum { T = %(T)d, B = %(B)d, H = %(H)d, D = %(D)d, STRIDE = %(STRIDE)d, R = 3, N = 6, ROWS = %(ROWS)d };
static const int32_t qsl[R + 1] = {%(QSL)s};
static const int64_t pos[N] = {%(POS)s};
static const int32_t table[R * STRIDE] = {%(TABLE)s};
static const int32_t g0[R] = {%(G0)s}, g1[R] = {%(G1)s};

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    printf("cuda error %%d at line %%d\n", (int)e_, __LINE__); return 2; } } while (0)

int main(void) {
    static uint16_t key[N * H * D], val[N * H * D], kout[ROWS * H * D], vout[ROWS * H * D];
    for (int i = 0; i < N * H * D; ++i) {
        key[i] = (uint16_t)(0x3c00 + i);
        val[i] = (uint16_t)(0x4000 + 3 * i);
    }
    const size_t cache_bytes = (size_t)B * T * H * D * 2;
    void *d_key, *d_val, *d_kc, *d_vc, *d_ko, *d_vo;
    int32_t *d_qsl, *d_table, *d_g0, *d_g1, *d_err;
    int64_t *d_pos, *d_slot;
    cudaStream_t s;
    CK(cudaStreamCreate(&s));
    CK(cudaMalloc(&d_key, sizeof key));
    CK(cudaMalloc(&d_val, sizeof val));
    CK(cudaMalloc(&d_kc, cache_bytes));
    CK(cudaMalloc(&d_vc, cache_bytes));
    CK(cudaMalloc(&d_ko, sizeof kout));
    CK(cudaMalloc(&d_vo, sizeof vout));
    CK(cudaMalloc((void**)&d_qsl, sizeof qsl));
    CK(cudaMalloc((void**)&d_table, sizeof table));
    CK(cudaMalloc((void**)&d_g0, sizeof g0));
    CK(cudaMalloc((void**)&d_g1, sizeof g1));
    CK(cudaMalloc((void**)&d_err, sizeof(int32_t)));
    CK(cudaMalloc((void**)&d_pos, sizeof pos));
    CK(cudaMalloc((void**)&d_slot, (N + 2) * sizeof(int64_t)));
    CK(cudaMemcpy(d_key, key, sizeof key, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_val, val, sizeof val, cudaMemcpyHostToDevice));
    CK(cudaMemset(d_kc, 0, cache_bytes));
    CK(cudaMemset(d_vc, 0, cache_bytes));
    CK(cudaMemcpy(d_qsl, qsl, sizeof qsl, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_pos, pos, sizeof pos, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_table, table, sizeof table, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_g0, g0, sizeof g0, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_g1, g1, sizeof g1, cudaMemcpyHostToDevice));
    CK(cudaMemset(d_err, 0, sizeof(int32_t)));

    int rc = kv_slot_mapping_paged_write(d_qsl, d_pos, d_table, STRIDE, R, N, N + 2, T, B,
                                         d_key, d_val, d_kc, d_vc, 1, H, D, d_slot, d_err,
                                         (kv_stream_t)s);
    if (rc != KV_OK) { printf("write: %%s\n", kv_status_string(rc)); return 3; }
    rc = kv_cache_gather(d_kc, d_vc, 0, 1, B, T, H, D, d_table, STRIDE, d_g0, d_g1, R, d_ko,
                         d_vo, ROWS, d_err, (kv_stream_t)s);
    if (rc != KV_OK) { printf("gather: %%s\n", kv_status_string(rc)); return 3; }
    CK(cudaStreamSynchronize(s));

    int64_t slot[N + 2];
    int32_t err;
    CK(cudaMemcpy(slot, d_slot, sizeof slot, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&err, d_err, sizeof err, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(kout, d_ko, sizeof kout, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(vout, d_vo, sizeof vout, cudaMemcpyDeviceToHost));
    printf("slots");
    for (int i = 0; i < N + 2; ++i) printf(" %%lld", (long long)slot[i]);
    printf("\nerr %%d\nk", (int)err);
    for (int i = 0; i < ROWS * H * D; ++i) printf(" %%u", (unsigned)kout[i]);
    printf("\nv");
    for (int i = 0; i < ROWS * H * D; ++i) printf(" %%u", (unsigned)vout[i]);
    printf("\n");
    return 0;
}
"""


def _expected():
    N = len(POS)
    rows = sum(b - a for a, b in zip(G0, G1))
    key = np.array([0x3c00 + i for i in range(N * H * D)], np.uint16).reshape(1, N, H, D)
    val = np.array([0x4000 + 3 * i for i in range(N * H * D)], np.uint16).reshape(1, N, H, D)
    table = np.array(TABLE, np.int32)
    slots, e1 = oracle.slot_mapping_paged(QSL, POS, table, N, N + 2, T, B)
    kc = np.zeros((1, B, T, H, D), np.uint16)
    vc = np.zeros_like(kc)
    e2 = oracle.cache_write(key, val, kc, vc, slots[:N], B, T)
    ko = np.zeros((rows, H, D), np.uint16)
    vo = np.zeros_like(ko)
    e3 = oracle.cache_gather(kc, vc, 0, B, T, table, G0, G1, ko, vo)
    return slots, e1 | e2 | e3, ko.reshape(-1), vo.reshape(-1), rows


def test_c_program_on_the_gpu(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    slots, err, ko, vo, rows = _expected()
    join = lambda xs: ", ".join(str(int(x)) for x in xs)  # noqa: E731
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM % dict(T=T, B=B, H=H, D=D, STRIDE=STRIDE, ROWS=rows, QSL=join(QSL),
                                  POS=join(POS), TABLE=join(np.array(TABLE).reshape(-1)),
                                  G0=join(G0), G1=join(G1)))
    exe = tmp_path / "consumer"
    from paged_kv_cache_39_gb300 import _lib
    assert os.path.exists(_lib.LIB_PATH), "build the library first"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), str(src), "-o", str(exe), "-L", PKG, "-lkvpaged",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{PKG}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    out = {line.split()[0]: line.split()[1:] for line in r.stdout.splitlines() if line.strip()}
    assert [int(x) for x in out["slots"]] == slots.tolist()
    assert int(out["err"][0]) == err
    assert np.array_equal(np.array(out["k"], np.int64), ko.astype(np.int64))
    assert np.array_equal(np.array(out["v"], np.int64), vo.astype(np.int64))
