"""Compile the CPU oracle (``pa_oracle.c``) into ``oracle/_build/liboracle.so``.

Test infrastructure: the product never loads this library.  Plain gcc, fp64,
no fused multiply-add contraction, so the arithmetic is the one the C source
spells out on both x86 and Arm hosts.
"""
from __future__ import annotations

import os
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
SRC = HERE / "pa_oracle.c"
OUT_DIR = HERE / "_build"
LIB = OUT_DIR / "liboracle.so"


def build(force: bool = False) -> Path:
    OUT_DIR.mkdir(exist_ok=True)
    if not force and LIB.exists() and LIB.stat().st_mtime >= SRC.stat().st_mtime:
        return LIB
    tmp = OUT_DIR / f"liboracle.{os.getpid()}.so"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", str(tmp), str(SRC), "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def build_from_text(source: str, name: str) -> Path:
    """Compile a modified copy of the oracle source (the CPU tests plant a
    mistake in such a copy to show that the pins catch it)."""
    OUT_DIR.mkdir(exist_ok=True)
    src = OUT_DIR / f"pa_oracle_{name}.c"
    src.write_text(source)
    out = OUT_DIR / f"liboracle_{name}.so"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", str(out), str(src), "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    print(build(force=True))
