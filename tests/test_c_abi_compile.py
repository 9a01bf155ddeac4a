"""The C ABI from C: include/rmsnorm.h compiles as C11 and as C++17, before
or after the CUDA runtime header, and a C program linked against the library
gets the status codes the header documents for argument errors (checked
before any CUDA call, so this runs without a GPU)."""
import os
import shutil
import subprocess

import pytest

from tests.conftest import ROOT

INCLUDE = os.path.join(ROOT, "include")
CUDA_INCLUDE = "/usr/local/cuda/include"

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#if CUDA_FIRST
#include <cuda_runtime_api.h>
#endif
#include "rmsnorm.h"
#if !CUDA_FIRST && WITH_CUDA
#include <cuda_runtime_api.h>
#endif

int main(void) {
  int bad = 0;
  /* a NULL input is an argument error, reported before any CUDA call */
  float rstd[4];
  rmsnorm_status_t s = rmsnorm_fwd(NULL, NULL, NULL, rstd, 4, 8, 1e-6f, RMSNORM_BF16,
                                   RMSNORM_BF16, (cudaStream_t)0);
  if (s != RMSNORM_ERR_INVALID_ARG) { printf("fwd NULL: %d\n", (int)s); bad = 1; }
  /* negative sizes and a negative eps */
  s = rmsnorm_fwd(rstd, rstd, rstd, NULL, -1, 8, 1e-6f, RMSNORM_F32, RMSNORM_F32, 0);
  if (s != RMSNORM_ERR_INVALID_ARG) { printf("fwd M<0: %d\n", (int)s); bad = 1; }
  s = rmsnorm_fwd(rstd, rstd, rstd, NULL, 1, 4, -1.f, RMSNORM_F32, RMSNORM_F32, 0);
  if (s != RMSNORM_ERR_INVALID_ARG) { printf("fwd eps<0: %d\n", (int)s); bad = 1; }
  /* an unsupported dtype pair */
  s = rmsnorm_fwd(rstd, rstd, rstd, NULL, 1, 4, 1e-6f, RMSNORM_F32, RMSNORM_BF16, 0);
  if (s != RMSNORM_ERR_UNSUPPORTED_DTYPE) { printf("fwd pair: %d\n", (int)s); bad = 1; }
  /* no rows: nothing to do */
  s = rmsnorm_fwd(NULL, NULL, NULL, NULL, 0, 8, 1e-6f, RMSNORM_BF16, RMSNORM_BF16, 0);
  if (s != RMSNORM_OK) { printf("fwd M=0: %d\n", (int)s); bad = 1; }
  if (strcmp(rmsnorm_status_string(RMSNORM_OK), "ok") != 0) { printf("string\n"); bad = 1; }
  if (rmsnorm_status_string((rmsnorm_status_t)99) == NULL) { printf("string 99\n"); bad = 1; }
  printf(bad ? "FAIL\n" : "PASS\n");
  return bad;
}
"""


def _lib():
    from row_wise_normalization_02_gb300 import _build
    return _build.build()


@pytest.mark.parametrize("lang,std", [("c", "c11"), ("c++", "c++17")])
@pytest.mark.parametrize("cuda_first,with_cuda", [(0, 0), (1, 1), (0, 1)])
def test_header_compiles_and_reports_argument_errors(tmp_path, lang, std, cuda_first, with_cuda):
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    if with_cuda and not os.path.exists(os.path.join(CUDA_INCLUDE, "cuda_runtime_api.h")):
        pytest.skip("no CUDA runtime header")
    lib = _lib()
    src = tmp_path / ("prog.c" if lang == "c" else "prog.cpp")
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    cmd = [cc, f"-std={std}", "-Wall", "-Wextra", "-Werror", f"-DCUDA_FIRST={cuda_first}",
           f"-DWITH_CUDA={with_cuda}", "-I", INCLUDE, "-I", CUDA_INCLUDE, str(src),
           "-o", str(exe), lib, f"-Wl,-rpath,{os.path.dirname(lib)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and "PASS" in out.stdout, out.stdout + out.stderr
