"""Build the host and device generator libraries in-tree."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build_host() -> str:
    out = os.path.join(_HERE, "libcsa2synth_host.so")
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared", "-pthread",
           os.path.join(_HERE, "synth_host.c"), "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build_dev_cmd() -> list[str]:
    out = os.path.join(_HERE, "libcsa2synth_dev.so")
    return ["nvcc", *NVCC_ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-shared",
            "-Xcompiler", "-fPIC", "-cudart", "static", os.path.join(_HERE, "synth_dev.cu"),
            "-o", out]


def build_dev() -> str:
    cmd = build_dev_cmd()
    subprocess.run(cmd, check=True)
    return cmd[-1]
