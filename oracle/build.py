"""Compile the C oracle (test infrastructure) with gcc into oracle/libfp8z_oracle.so."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def oracle_lib_path() -> str:
    return os.path.join(_HERE, "libfp8z_oracle.so")


def build_oracle(force: bool = False) -> str:
    src = os.path.join(_HERE, "fp8z_oracle.c")
    out = oracle_lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off: no FMA contraction (gcc contracts by default on aarch64);
    # IEEE division and sqrtf; no fast-math.
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(force=True))
