"""Build the CPU oracle's shared library with the host compiler only.

    python -m oracle.build

Compiles moe_oracle.cpp (plain single-threaded C++17, no GPU code, no
-march: the library is built on one machine and may run on another) into
oracle/libmoe_oracle.so.  Test infrastructure: nothing in the CUDA library
links or calls it.
"""

from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
HDR = os.path.join(HERE, "moe_oracle.h")
LIB = os.path.join(HERE, "libmoe_oracle.so")


def build(force: bool = False) -> str:
    """Path of the oracle library, compiled if missing or older than its
    sources.  MOE_ORACLE_LIB names a prebuilt one instead (for example an
    AddressSanitizer build)."""
    if os.environ.get("MOE_ORACLE_LIB"):
        return os.environ["MOE_ORACLE_LIB"]
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) > newest:
        return LIB
    cxx = os.environ.get("CXX", "g++")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cxx, "-std=c++17", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)            # atomic: a concurrent loader sees old or new
    return LIB


if __name__ == "__main__":
    print(build(force=True))
