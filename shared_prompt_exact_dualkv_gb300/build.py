"""Builds libdualkv.so in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel to an object file, then one link
step produces the shared library next to this file.  Run as
``python -m shared_prompt_exact_dualkv_gb300.build`` or through
``__graft_entry__.build()``.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libdualkv.so")
# the checks build: device-side index and pipeline checks (-DDUALKV_CHECKS)
CHECKS_BUILD_DIR = os.path.join(HERE, "_build_checks")
CHECKS_LIB_PATH = os.path.join(HERE, "libdualkv_checks.so")

SOURCES = ["api.cu", "fwd.cu", "dq.cu", "dkdv.cu", "small.cu", "layer_kernels.cu", "layer_api.cu", "gemm.cu"]
LIBS = []
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, extra: list, build_dir: str = BUILD_DIR) -> tuple:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def build(verbose: bool = False, extra=None, checks: bool = False) -> str:
    """Compile every CUDA source and link libdualkv.so (or, with checks=True,
    the checks build libdualkv_checks.so); returns its path."""
    extra = list(extra or [])
    build_dir, lib_path = BUILD_DIR, LIB_PATH
    if checks:
        extra.append("-DDUALKV_CHECKS")
        build_dir, lib_path = CHECKS_BUILD_DIR, CHECKS_LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    logs = []
    for src, obj, rc, log in results:
        logs.append(f"== {src}\n{log}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{log}")
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    objs = [r[1] for r in results]
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, *LIBS]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, lib_path)
    if verbose:
        print("\n".join(logs))
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, checks="--checks" in sys.argv))
