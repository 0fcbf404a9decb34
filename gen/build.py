"""Builds the host (gcc) and device (nvcc, sm_103a) copies of the generator."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _newer(out: str, srcs) -> bool:
    return os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(s) for s in srcs)


def build_host() -> str:
    out = os.path.join(HERE, "libmoegen_host.so")
    srcs = [os.path.join(HERE, "moegen_host.c"), os.path.join(HERE, "moegen.h")]
    if not _newer(out, srcs):
        base = ["gcc", "-O2", "-shared", "-fPIC", "-o", out, srcs[0]]
        try:
            subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True)
    return out


def build_dev() -> str:
    out = os.path.join(HERE, "libmoegen_dev.so")
    srcs = [os.path.join(HERE, "moegen_dev.cu"), os.path.join(HERE, "moegen.h")]
    if not _newer(out, srcs):
        subprocess.run([NVCC, "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                        "-Xcompiler", "-fPIC", "-o", out, srcs[0]], check=True)
    return out


def build() -> None:
    build_host()
    build_dev()
