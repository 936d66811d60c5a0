"""Compile the C oracle into ``oracle/libkvoracle.so`` with the host C compiler.

Test infrastructure: building the checker is part of the build step, using it
is reserved to the tests, the smoke check and the benchmark's CPU baseline.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "kv_oracle.c")


def library_path(variant: str = "") -> str:
    return os.path.join(HERE, f"libkvoracle{variant}.so")


def build_oracle(extra_flags=(), variant: str = "", source: str = SOURCE, out: str = None) -> str:
    """Build the oracle shared library; returns its path."""
    out = out or library_path(variant)
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-fPIC", "-shared",
           *extra_flags, source, "-o", out + ".tmp"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build_oracle(sys.argv[1:]))
