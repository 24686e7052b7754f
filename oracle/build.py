"""Compile the fp64 CPU oracle (``bi_oracle.c``) into a shared library.

Test infrastructure: the oracle is built so the tests, the smoke check and the
benchmark's CPU-baseline leg can call it; the product never loads it.

Flags: ``-O2 -fno-fast-math -ffp-contract=off`` keep every double operation a
separately rounded IEEE operation (no fused multiply-add contraction, no
reassociation).  OpenMP is used when the compiler supports it; it only spreads
independent outputs over threads.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bi_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

BASE_FLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
              "-std=c11", "-Wall"]


def _compile(extra: list[str], out: str) -> subprocess.CompletedProcess:
    cmd = ["gcc", *BASE_FLAGS, *extra, SRC, "-o", out, "-lm"]
    return subprocess.run(cmd, capture_output=True, text=True)


def build_oracle(force: bool = False) -> str:
    """Build ``_build/liboracle.so`` if missing or older than the source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    # write to a temp name and rename, so concurrent builders never see a
    # half-written library
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=OUT_DIR)
    os.close(fd)
    r = _compile(["-fopenmp"], tmp)
    if r.returncode != 0:
        r = _compile([], tmp)
    if r.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
