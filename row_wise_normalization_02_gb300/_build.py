"""Build librmsnorm_gb300.so in-tree with nvcc for sm_103a.

Twenty-eight translation units (forward, backward, staged, ragged, mixed-alignment
ragged, cluster, wide, quantised-output and LayerNorm kernels once per dtype pair,
plus the C ABI)
compile in parallel, then link into one shared library with the CUDA runtime
linked statically.  Rebuilds only when a source is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIB = os.path.join(PKG, "librmsnorm_gb300.so")
OBJDIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr"]

UNITS = [("rmsnorm_fwd.cu", ["-DRMSN_PAIR=0"], "fwd_p0.o"),
         ("rmsnorm_fwd.cu", ["-DRMSN_PAIR=1"], "fwd_p1.o"),
         ("rmsnorm_fwd.cu", ["-DRMSN_PAIR=2"], "fwd_p2.o"),
         ("rmsnorm_bwd.cu", ["-DRMSN_PAIR=0"], "bwd_p0.o"),
         ("rmsnorm_bwd.cu", ["-DRMSN_PAIR=1"], "bwd_p1.o"),
         ("rmsnorm_bwd.cu", ["-DRMSN_PAIR=2"], "bwd_p2.o"),
         ("rmsnorm_staged.cu", ["-DRMSN_PAIR=0"], "staged_p0.o"),
         ("rmsnorm_staged.cu", ["-DRMSN_PAIR=1"], "staged_p1.o"),
         ("rmsnorm_staged.cu", ["-DRMSN_PAIR=2"], "staged_p2.o"),
         ("rmsnorm_ragged.cu", ["-DRMSN_PAIR=0"], "ragged_p0.o"),
         ("rmsnorm_ragged.cu", ["-DRMSN_PAIR=1"], "ragged_p1.o"),
         ("rmsnorm_ragged.cu", ["-DRMSN_PAIR=2"], "ragged_p2.o"),
         ("rmsnorm_ragged.cu", ["-DRMSN_PAIR=0", "-DRMSN_MIX=1"], "ragged_mix_p0.o"),
         ("rmsnorm_ragged.cu", ["-DRMSN_PAIR=1", "-DRMSN_MIX=1"], "ragged_mix_p1.o"),
         ("rmsnorm_ragged.cu", ["-DRMSN_PAIR=2", "-DRMSN_MIX=1"], "ragged_mix_p2.o"),
         ("rmsnorm_quant.cu", ["-DRMSN_PAIR=0"], "quant_p0.o"),
         ("rmsnorm_quant.cu", ["-DRMSN_PAIR=1"], "quant_p1.o"),
         ("rmsnorm_quant.cu", ["-DRMSN_PAIR=2"], "quant_p2.o"),
         ("rmsnorm_layernorm.cu", ["-DRMSN_PAIR=0"], "ln_p0.o"),
         ("rmsnorm_layernorm.cu", ["-DRMSN_PAIR=1"], "ln_p1.o"),
         ("rmsnorm_layernorm.cu", ["-DRMSN_PAIR=2"], "ln_p2.o"),
         ("rmsnorm_cluster.cu", ["-DRMSN_PAIR=0"], "cluster_p0.o"),
         ("rmsnorm_cluster.cu", ["-DRMSN_PAIR=1"], "cluster_p1.o"),
         ("rmsnorm_cluster.cu", ["-DRMSN_PAIR=2"], "cluster_p2.o"),
         ("rmsnorm_wide.cu", ["-DRMSN_PAIR=0"], "wide_p0.o"),
         ("rmsnorm_wide.cu", ["-DRMSN_PAIR=1"], "wide_p1.o"),
         ("rmsnorm_wide.cu", ["-DRMSN_PAIR=2"], "wide_p2.o"),
         ("rmsnorm_api.cu", [], "api.o")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources():
    out = [os.path.join(INCLUDE, "rmsnorm.h")]
    for f in os.listdir(CSRC):
        out.append(os.path.join(CSRC, f))
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources()) and os.path.getmtime(__file__) <= t


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    cc = nvcc()

    def compile_unit(u):
        src, defs, obj = u
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, *defs, "-I", INCLUDE, "-c",
               os.path.join(CSRC, src), "-o", os.path.join(OBJDIR, obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src} {defs}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(UNITS), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = f"{LIB}.{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[os.path.join(OBJDIR, o) for o in objs],
           "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
