"""The boundary from C: include/ozk.h compiles as strict C99 and as C++17,
and a C program that takes the address of every entry point the header
declares links against libozk.so and, with no GPU, gets the same answers
from the host-only helpers and the argument checks as the Python binding
does.  (A declaration that does not match an exported symbol fails the
link.)"""
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
