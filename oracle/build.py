"""Builds the CPU oracle (test infrastructure) into oracle/_build/libkda_oracle.so.

Plain g++ in double precision: -O2 without -ffast-math or -march flags, so the same
source gives the same results on x86_64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_oracle.cpp")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkda_oracle.so")


def compile_source(src: str, out: str) -> str:
    """Compiles one oracle source file into a shared library at `out` (the flags above)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp]
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_source(SRC, LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
