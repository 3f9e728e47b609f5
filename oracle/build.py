"""Build the oracle library (plain C, -O2 -ffp-contract=off) in-tree."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def build() -> str:
    out = os.path.join(_HERE, "libcsa2oracle.so")
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-Wall", "-Wno-unused-function", os.path.join(_HERE, "csa2_oracle.c"), "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out
