"""Build step for the CPU oracle: compiles ``iso_oracle.c`` into a shared
library beside it with the system C compiler (portable C11, no ISA flags, so
it builds the same on x86_64 and aarch64)."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def build(verbose: bool = False) -> str:
    src = os.path.join(_HERE, "iso_oracle.c")
    out = library_path()
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, src, "-lm", "-lpthread"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
