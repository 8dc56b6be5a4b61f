"""The boundary from C: include/ozk.h compiles as strict C99 and as C++17,
and a C program that takes the address of every entry point the header
declares links against libozk.so and, with no GPU, gets the same answers
from the host-only helpers and the argument checks as the Python binding
does.  (A declaration that does not match an exported symbol fails the
link.)  On a GPU, a C program with device buffers from the CUDA runtime
gets C bit-exact from ozk_dgemm and ozk_dgemm_host."""
import os
import re
import shutil
import subprocess

import pytest

import oracle
from fp64_gemm_emulation_exponent_gb300 import build as ozk_build
from fp64_gemm_emulation_exponent_gb300 import ozk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
HEADER = os.path.join(INCLUDE, "ozk.h")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None or shutil.which("g++") is None,
                                reason="needs gcc and g++")


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(ozk_[a-z0-9_]+)\s*\(", text)))


def compile_ok(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_header_is_strict_c99_and_cxx17(tmp_path):
    src = tmp_path / "only_header.c"
    src.write_text('#include "ozk.h"\nint ozk_header_probe(void) { return OZK_MAX_MODULI; }\n')
    compile_ok(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, "-c", str(src),
                "-o", str(tmp_path / "c.o")])
    cxx = tmp_path / "only_header.cc"
    cxx.write_text('#include "ozk.h"\nint ozk_header_probe() { return OZK_MAX_MODULI; }\n')
    compile_ok(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-c", str(cxx),
                "-o", str(tmp_path / "cc.o")])


def test_c_program_links_every_entry_point_and_runs_without_a_gpu(tmp_path):
    lib = ozk_build.build()
    names = declared_functions()
    table = ",\n  ".join(f"(any_fn){n}" for n in names)
    src = tmp_path / "caller.c"
    src.write_text(f"""#include <stdio.h>
#include "ozk.h"

typedef void (*any_fn)(void);
static const any_fn entry_points[] = {{
  {table}
}};

int main(void) {{
  int32_t m[OZK_MAX_MODULI];
  double a[4] = {{0}}, b[4] = {{0}}, c[4] = {{0}};
  ozk_workspace_info info;
  int k;
  printf("%d\\n", (int)(sizeof entry_points / sizeof entry_points[0]));
  printf("%d\\n", ozk_moduli(OZK_MAX_MODULI, m));
  for (k = 0; k < OZK_MAX_MODULI; ++k) printf("%d ", m[k]);
  printf("\\n%d %d %d\\n", ozk_beta(4096, 14), ozk_gamma(4096, 13), ozk_moduli_for_bits(4096, 53));
  printf("%lld\\n", (long long)ozk_kpad(1000));
  printf("%lu\\n", (unsigned long)ozk_workspace_size(4096, 4096, 4096, 14));
  k = ozk_workspace_layout(4096, 4096, 4096, 14, &info);
  printf("%d %d %lu\\n", k, info.splits, (unsigned long)info.total_bytes);
  printf("%s\\n", ozk_status_string(OZK_ERR_TIMEOUT));
  printf("%d\\n", ozk_dgemm(-1, 2, 2, a, 2, b, 2, c, 2, 14, NULL));
  printf("%d\\n", ozk_dgemm(2, 2, 2, a, 2, b, 2, c, 2, 21, NULL));
  printf("%d\\n", ozk_dgemm(2, 2, 2, a, 2, b, 2, a, 2, 14, NULL));
  printf("%d\\n", ozk_dgemm(0, 5, 3, NULL, 3, NULL, 5, NULL, 5, 14, NULL));
  return 0;
}}
""")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(lib)
    compile_ok(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, str(src), "-L", libdir,
                "-lozk", f"-Wl,-rpath,{libdir}", "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out = r.stdout.splitlines()
    assert int(out[0]) == len(names)
    assert int(out[1]) == ozk.OZK_OK
    assert [int(x) for x in out[2].split()] == [int(p) for p in oracle.moduli(20)]
    beta, gamma, nbits = (int(x) for x in out[3].split())
    assert beta == ozk.ozk_beta(4096, 14) == oracle.beta(4096, 14)
    assert gamma == ozk.ozk_gamma(4096, 13) == oracle.gamma(4096, 13)
    assert nbits == ozk.ozk_moduli_for_bits(4096, 53)
    assert int(out[4]) == ozk.ozk_kpad(1000)
    assert int(out[5]) == ozk.ozk_workspace_size(4096, 4096, 4096, 14)
    status, splits, total = (int(x) for x in out[6].split())
    assert status == ozk.OZK_OK and splits >= 1 and total == int(out[5])
    assert out[7] == ozk.status_string(ozk.OZK_ERR_TIMEOUT)
    assert [int(x) for x in out[8:12]] == [ozk.OZK_ERR_INVALID_ARG, ozk.OZK_ERR_UNSUPPORTED,
                                           ozk.OZK_ERR_INVALID_ARG, ozk.OZK_OK]


@pytest.mark.gpu
def test_c_program_multiplies_on_the_gpu(tmp_path):
    """A plain C caller (CUDA runtime for device memory, no Python in the
    loop): ozk_dgemm on device buffers and ozk_dgemm_host on host buffers,
    both bit-exact against the oracle."""
    import numpy as np

    lib = ozk_build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    M, N, K, n = 67, 45, 130, 14
    rng = np.random.default_rng(5)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    A.tofile(tmp_path / "a.bin")
    B.tofile(tmp_path / "b.bin")
    src = tmp_path / "gpu_caller.c"
    src.write_text(f"""#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "ozk.h"

static int load(const char* path, double* x, size_t count) {{
  FILE* f = fopen(path, "rb");
  size_t got;
  if (!f) return 1;
  got = fread(x, sizeof(double), count, f);
  fclose(f);
  return got != count;
}}

int main(int argc, char** argv) {{
  const int64_t M = {M}, N = {N}, K = {K};
  double *A = malloc(sizeof(double) * M * K), *B = malloc(sizeof(double) * K * N);
  double *C1 = malloc(sizeof(double) * M * N), *C2 = malloc(sizeof(double) * M * N);
  double *dA, *dB, *dC;
  int rc, i;
  if (argc < 3 || load(argv[1], A, M * K) || load(argv[2], B, K * N)) return 10;
  if (cudaMalloc((void**)&dA, sizeof(double) * M * K) || cudaMalloc((void**)&dB, sizeof(double) * K * N) ||
      cudaMalloc((void**)&dC, sizeof(double) * M * N))
    return 11;
  cudaMemcpy(dA, A, sizeof(double) * M * K, cudaMemcpyHostToDevice);
  cudaMemcpy(dB, B, sizeof(double) * K * N, cudaMemcpyHostToDevice);
  rc = ozk_dgemm(M, N, K, dA, K, dB, N, dC, N, {n}, NULL);
  if (rc != OZK_OK) return 20 + rc;
  if (ozk_stream_status(NULL) != OZK_OK) return 14;  /* waits for the call */
  if (cudaMemcpy(C1, dC, sizeof(double) * M * N, cudaMemcpyDeviceToHost)) return 12;
  rc = ozk_dgemm_host(M, N, K, A, K, B, N, C2, N, {n}, NULL);
  if (rc != OZK_OK) return 30 + rc;
  if (ozk_stream_status(NULL) != OZK_OK) return 13;
  for (i = 0; i < M * N; ++i) printf("%a %a\\n", C1[i], C2[i]);
  cudaFree(dA);
  cudaFree(dB);
  cudaFree(dC);
  free(A); free(B); free(C1); free(C2);
  return 0;
}}
""")
    exe = tmp_path / "gpu_caller"
    libdir = os.path.dirname(lib)
    compile_ok(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-I", os.path.join(cuda, "include"),
                str(src), "-L", libdir, "-lozk", f"-Wl,-rpath,{libdir}", "-L", os.path.join(cuda, "lib64"),
                "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", str(exe)])
    r = subprocess.run([str(exe), str(tmp_path / "a.bin"), str(tmp_path / "b.bin")], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, (r.returncode, r.stderr)
    got = np.array([[float.fromhex(v) for v in line.split()] for line in r.stdout.splitlines()])
    want = oracle.dgemm(A, B, n).ravel()
    assert got.shape == (M * N, 2)
    assert np.array_equal(got[:, 0].view(np.uint64), want.view(np.uint64))
    assert np.array_equal(got[:, 1].view(np.uint64), want.view(np.uint64))
