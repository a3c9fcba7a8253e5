"""Compile the C++ CPU oracle into ``oracle/libdsa_oracle.so``.

Plain ``g++ -O2 -std=c++17 -fopenmp -shared -fPIC`` of ``dsa_oracle.cpp``; no
architecture-specific flags, so the same source builds on x86-64 and Arm
hosts. Rebuilt when the source is newer than the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dsa_oracle.cpp")
LIB = os.path.join(HERE, "libdsa_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC", "-Wall"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("no C++ compiler found to build the CPU oracle")
    tmp = f"{LIB}.{os.getpid()}.tmp"
    r = subprocess.run([cxx, *FLAGS, SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the CPU oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
