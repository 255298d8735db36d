"""Build the fp64 CPU oracle (plain C, gcc, OpenMP) into a shared library.

Test infrastructure: the oracle is built next to its source and loaded only by
the tests, the smoke check and the benchmark's CPU-baseline leg.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mlstm_oracle.c")


def lib_path(mutation: int = 0) -> str:
    name = "libmlstm_oracle.so" if mutation == 0 else f"libmlstm_oracle_mut{mutation}.so"
    return os.path.join(HERE, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally with planted mistake `mutation`)."""
    out = lib_path(mutation)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = f"{out}.tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           f"-DORACLE_MUTATION={int(mutation)}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)            # atomic: concurrent builders never see a partial file
    return out


if __name__ == "__main__":
    muts = [int(a) for a in sys.argv[1:]] or [0]
    for m in muts:
        print(build(m, force=True))
