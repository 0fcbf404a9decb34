"""Compiles the C oracle (test infrastructure) with gcc; OpenMP when available."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT = os.path.join(HERE, "liboracle.so")


def build() -> str:
    if os.path.exists(OUT) and os.path.getmtime(OUT) >= os.path.getmtime(SRC):
        return OUT
    # -ffp-contract=off: no fused multiply-add may change a rounding of the oracle
    base = ["gcc", "-O2", "-ffp-contract=off", "-shared", "-fPIC", "-o", OUT, SRC, "-lm"]
    try:
        subprocess.run(base[:3] + ["-fopenmp"] + base[3:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    return OUT
