"""Compile the CPU oracle (TEST INFRASTRUCTURE ONLY) into oracle/liboracle.so.

Flags: -O2, -ffp-contract=off (no fused multiply-add, which GCC emits by default on
aarch64), no -ffast-math, no -march=native, so the same source gives the same bits on
x86_64 and aarch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "liboracle.so")
SOURCES = [os.path.join(HERE, "oracle.cpp")]
FLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
         "-Wall", "-Wextra"]


def build(force=False):
    newest = max(os.path.getmtime(p) for p in SOURCES + [os.path.join(HERE, "oracle.h")])
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["g++"] + FLAGS + SOURCES + ["-o", tmp])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
