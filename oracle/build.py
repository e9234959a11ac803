"""Compile oracle.c into liboracle.so with the system C compiler (test infrastructure)."""

from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def source_path() -> str:
    return os.path.join(_HERE, "oracle.c")


def library_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def build() -> str:
    out = library_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", source_path(), "-lm", "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build())
