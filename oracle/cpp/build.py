"""Build the C++ oracle: oracle/cpp/moe_oracle.cpp -> oracle/cpp/_build/libmoe_oracle.so.

Plain g++ (C++17, -O2, -ffp-contract=off so that no multiply-add is fused and
every floating-point step rounds as written, -pthread for std::thread).
Test infrastructure: only the tests and the CPU-baseline leg of bench.py load
the result.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libmoe_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    stamp = os.path.join(OUT, "host_arch")
    arch = platform.machine()
    stale = (force or not os.path.exists(LIB) or os.path.getmtime(SRC) > os.path.getmtime(LIB)
             or not os.path.exists(stamp) or open(stamp).read().strip() != arch)
    if stale:
        cxx = shutil.which("g++") or shutil.which("c++")
        if cxx is None:
            raise RuntimeError("g++ not found: needed to build the C++ oracle")
        tmp = LIB + ".tmp%d" % os.getpid()
        r = subprocess.run([cxx, *FLAGS, "-o", tmp, SRC], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
        os.replace(tmp, LIB)
        with open(stamp, "w") as f:
            f.write(arch)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
