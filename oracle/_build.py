"""Compile the C oracle into ``oracle/liboracle.so`` (plain gcc, no fast-math,
no FMA contraction, so the binary64 arithmetic is the same on x86-64 and
aarch64)."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    out = library_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out
