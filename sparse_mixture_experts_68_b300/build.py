"""Build libmoe.so in-tree with nvcc for sm_103a.

    python -m sparse_mixture_experts_68_b300.build [--checks] [--ptxas]

Each .cu under csrc/ compiles to an object in _build/ (in parallel), then one
shared library is linked next to this file.  ``--checks`` builds the checks
variant instead, libmoe_checks.so (objects in _build/checks/): -DMOE_CHECKS
turns on the kernels' index checks and the workspace guard gaps; the binding
loads it when MOE_LIBRARY=checks.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe.so")
LIB_CHECKS = os.path.join(PKG, "libmoe_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, ptxas_verbose: bool = False, checks: bool = False) -> str:
    out_dir = os.path.join(BUILD, "checks") if checks else BUILD
    lib_path = LIB_CHECKS if checks else LIB
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if checks:
        flags.append("-DMOE_CHECKS")
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "moe.h"))
    newest_header = max(os.path.getmtime(h) for h in headers)

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        if (not ptxas_verbose and os.path.exists(obj)
                and os.path.getmtime(obj) > max(os.path.getmtime(src), newest_header)):
            return obj, ""
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for _, log in results:
            if log:
                print(log)
    objs = [o for o, _ in results]
    cmd = [nvcc] + ARCH + ["-shared", "-o", lib_path] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="--ptxas" in sys.argv, checks="--checks" in sys.argv))
