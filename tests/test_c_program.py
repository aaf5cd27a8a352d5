"""The C ABI used from a plain C program, with no Python between it and the library.

The program allocates device memory with the CUDA runtime's C API, plans and runs
a ragged CTA-pair GEMM on small-integer operands, reads the status and checks every
output against its own integer products, repeats it with two pairs sharing B
through multicast, then exercises the error paths a C caller meets.  Integer inputs make the expected values exact.
"""

import os
import shutil
import subprocess

import pytest

import software_pipelined_tiled_02_gb300 as tg
from software_pipelined_tiled_02_gb300 import build as tbuild
from tests.conftest import ROOT

C_PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "tgemm.h"

/* fp16 bits of a small integer |v| <= 2048 */
static uint16_t half_of_int(int v)
{
    if (v == 0) return 0;
    uint16_t sign = v < 0 ? 0x8000u : 0u;
    unsigned a = (unsigned)(v < 0 ? -v : v);
    int e = 0;
    while ((a >> e) > 1) ++e;
    unsigned mant = (a << (10 - e)) & 0x3FFu;
    return (uint16_t)(sign | (unsigned)((e + 15) << 10) | mant);
}

int main(void)
{
    const int M = 300, N = 520, K = 264;
    size_t na = (size_t)M * K, nb = (size_t)N * K, nc = (size_t)M * N;
    uint16_t *hA = malloc(na * 2), *hB = malloc(nb * 2);
    float *hC = malloc(nc * 4);
    int *iA = malloc(na * sizeof(int)), *iB = malloc(nb * sizeof(int));
    uint32_t x = 12345u;
    for (size_t i = 0; i < na; ++i) { x = x * 1664525u + 1013904223u; iA[i] = (int)((x >> 24) % 9u) - 4; hA[i] = half_of_int(iA[i]); }
    for (size_t i = 0; i < nb; ++i) { x = x * 1664525u + 1013904223u; iB[i] = (int)((x >> 24) % 9u) - 4; hB[i] = half_of_int(iB[i]); }

    void *dA = 0, *dB = 0, *dC = 0;
    if (cudaMalloc(&dA, na * 2) || cudaMalloc(&dB, nb * 2) || cudaMalloc(&dC, nc * 4)) { puts("cudaMalloc"); return 2; }
    cudaMemcpy(dA, hA, na * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dB, hB, nb * 2, cudaMemcpyHostToDevice);
    cudaMemset(dC, 0xFF, nc * 4);  /* NaN everywhere until the kernel writes */

    tgemm_plan_t plan = 0;
    tgemm_plan_opts opts;
    memset(&opts, 0, sizeof(opts));
    opts.cta_pair = 1;
    int rc = tgemm_plan_ex(&plan, M, N, K, TGEMM_F16, TGEMM_F32, 256, 224, 64, 4, &opts);
    if (rc != TGEMM_OK) { printf("plan: %s\n", tgemm_strerror(rc)); return 3; }
    rc = tgemm_run(plan, dA, dB, dC, 0);
    if (rc != TGEMM_OK) { printf("run: %s\n", tgemm_strerror(rc)); return 4; }
    cudaDeviceSynchronize();
    int detail[4] = {0, 0, 0, 0};
    rc = tgemm_status(plan, detail);
    if (rc != TGEMM_OK) { printf("status: %s\n", tgemm_strerror(rc)); return 5; }
    cudaMemcpy(hC, dC, nc * 4, cudaMemcpyDeviceToHost);
    long bad = 0;
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) {
            long s = 0;
            for (int k = 0; k < K; ++k) s += (long)iA[(size_t)i * K + k] * iB[(size_t)j * K + k];
            if (hC[(size_t)i * N + j] != (float)s) ++bad;
        }
    if (bad) { printf("%ld wrong outputs\n", bad); return 6; }

    /* the same product with two CTA pairs sharing B through multicast (clusters of four) */
    tgemm_plan_t mc = 0;
    opts.multicast_b = 1;
    rc = tgemm_plan_ex(&mc, M, N, K, TGEMM_F16, TGEMM_F32, 256, 352, 64, 4, &opts);
    if (rc != TGEMM_OK) { printf("multicast plan: %s\n", tgemm_strerror(rc)); return 11; }
    tgemm_plan_info info;
    if (tgemm_get_plan_info(mc, &info) != TGEMM_OK || info.multicast_b != 1 || info.grid % 4 != 0) { puts("info"); return 12; }
    cudaMemset(dC, 0xFF, nc * 4);
    if (tgemm_run(mc, dA, dB, dC, 0) != TGEMM_OK) { puts("multicast run"); return 13; }
    cudaDeviceSynchronize();
    if (tgemm_status(mc, detail) != TGEMM_OK) { puts("multicast status"); return 14; }
    cudaMemcpy(hC, dC, nc * 4, cudaMemcpyDeviceToHost);
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) {
            long s = 0;
            for (int k = 0; k < K; ++k) s += (long)iA[(size_t)i * K + k] * iB[(size_t)j * K + k];
            if (hC[(size_t)i * N + j] != (float)s) ++bad;
        }
    if (bad) { printf("multicast: %ld wrong outputs\n", bad); return 15; }
    tgemm_destroy(mc);
    opts.cta_pair = 0;  /* B is shared between pairs only */
    tgemm_plan_t none = 0;
    if (tgemm_plan_ex(&none, M, N, K, TGEMM_F16, TGEMM_F32, 256, 352, 64, 4, &opts) != TGEMM_ERR_INVALID_ARG || none) {
        puts("multicast without pairs");
        return 16;
    }

    /* error paths: a NULL plan, a misaligned pointer, an over-budget config */
    if (tgemm_run(0, dA, dB, dC, 0) != TGEMM_ERR_INVALID_ARG) { puts("null plan"); return 7; }
    if (tgemm_run(plan, (char *)dA + 2, dB, dC, 0) != TGEMM_ERR_ALIGNMENT) { puts("alignment"); return 8; }
    tgemm_plan_t big = 0;
    if (tgemm_plan(&big, M, N, K, TGEMM_F16, TGEMM_F32, 256, 256, 64, 4) != TGEMM_ERR_SMEM_BUDGET || big) { puts("budget"); return 9; }
    if (tgemm_destroy(plan) != TGEMM_OK) { puts("destroy"); return 10; }
    cudaFree(dA); cudaFree(dB); cudaFree(dC);
    puts("ok");
    return 0;
}
"""


def compile_program(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src = tmp_path / "gemm.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "gemm"
    libdir = os.path.dirname(tg.LIB_PATH)
    cmd = [gcc, "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), str(src), "-L", libdir, "-ltgemm", "-L", os.path.join(cuda, "lib64"),
           "-lcudart", "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", str(exe)]
    out = subprocess.run(cmd, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    tbuild.build()
    compile_program(tmp_path)


@pytest.mark.gpu
def test_c_program_runs_a_gemm(tmp_path):
    tbuild.build()
    exe = compile_program(tmp_path)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and run.stdout.strip().endswith("ok"), run.stdout + run.stderr
