"""Compiles the C oracle into ``oracle/liboracle.so`` with gcc (test infrastructure).

Flags keep results identical on x86_64 and aarch64 hosts: ISO C, no
floating-point contraction into fused multiply-adds, no machine-specific
tuning.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")


def library_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    out = library_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out
