"""Builds the CPU oracle (plain C, gcc) into ``oracle/liboracle.so``.

Test infrastructure: the oracle is the checker for the CUDA library, never part
of it. ``build(mutant=n)`` compiles a copy with a deliberately planted mistake
into a separate file, for the test that shows the oracle's pins catch it.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")


def lib_path(mutant: int = 0, out_dir: str | None = None) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(out_dir or HERE, name)


def build(mutant: int = 0, out_dir: str | None = None, force: bool = False) -> str:
    out = lib_path(mutant, out_dir)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
