"""Compile the oracle's C part (test infrastructure) with gcc, in place."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "router_fp32.c")
    out = os.path.join(_HERE, "liboracle_router.so")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                           "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
