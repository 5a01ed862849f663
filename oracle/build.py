"""Compile the C oracle into a shared library with gcc.

Test infrastructure: only the tests, the package smoke check and the
benchmark's CPU-baseline leg use the oracle.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pkv_oracle.c")
LIBRARY = os.path.join(HERE, "libpkv_oracle.so")


def build(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Build ``output`` from ``source`` (plain C11, -O2, no vectorisation
    flags, nothing machine specific) unless it is already newer."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + ".tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, source]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


if __name__ == "__main__":
    print(build(force=True))
