"""Compile the CPU oracle (plain C, gcc) into a shared library beside its source.

Test infrastructure only. `-ffp-contract=off` keeps every fp64 operation
separately rounded, so the oracle computes the same values on x86-64 and
aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sgq_oracle.c")
LIB = os.path.join(HERE, "libsgq_oracle.so")


def compile_oracle(src: str, out: str) -> str:
    """Compile the oracle source `src` into the shared library `out` (the
    mutation tests build planted-mistake copies with the same flags)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror", "-ffp-contract=off",
           "-fno-fast-math", "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build_oracle(force: bool = False) -> str:
    """Build libsgq_oracle.so if it is missing or older than its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_oracle(SRC, LIB)


if __name__ == "__main__":
    print(build_oracle(force=True))
