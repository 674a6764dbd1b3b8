"""Build the C++ oracle (oracle/moe_oracle_ref.cpp) into a shared library with g++.

TEST INFRASTRUCTURE (see oracle/__init__.py). Plain host C++17 with OpenMP; no
CUDA, no BLAS, no machine-specific flags, and floating-point contraction off so
that the same source gives the same numbers on x86_64 and aarch64 hosts.

    python -m oracle.build [--mutant N]

``mutant`` > 0 builds a library with one planted mistake (for the pin tests).
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle_ref.cpp")
BUILD = os.path.join(HERE, "_build")
FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def lib_path(mutant: int = 0) -> str:
    return os.path.join(BUILD, "libmoe_oracle.so" if mutant == 0 else f"libmoe_oracle_mut{mutant}.so")


def cxx() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand:
            return cand
    raise RuntimeError("no C++ compiler found for the oracle")


def build(mutant: int = 0, force: bool = False) -> str:
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.abspath(__file__))):
        return out
    os.makedirs(BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = [cxx(), *FLAGS, f"-DORACLE_MUTANT={int(mutant)}", SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("building the C++ oracle failed")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--mutant", type=int, default=0)
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    print(build(a.mutant, a.force))
