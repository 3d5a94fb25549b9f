"""Build the CPU oracle (test infrastructure only).

``build()`` compiles ``ssd_oracle.c`` with gcc into ``libssd_oracle.so`` beside this
file: ``-O2 -ffp-contract=off`` (every double operation rounds once, as written, no
fast-math) and OpenMP over independent (sequence, head) units.  ``build(mutant=k)``
plants mutation k (1..9) and writes ``libssd_oracle_m{k}.so``; the mutation tests
use those to show that the oracle's pins fail on each planted mistake.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ssd_oracle.c")


def lib_path(mutant: int | None = None) -> str:
    name = "libssd_oracle.so" if not mutant else f"libssd_oracle_m{int(mutant)}.so"
    return os.path.join(HERE, name)


def build(mutant: int | None = None, force: bool = False) -> str:
    out = lib_path(mutant)
    hdr = os.path.join(HERE, "ssd_oracle.h")
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(SRC), os.path.getmtime(hdr))):
        return out
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall",
           "-Wextra", "-Werror", "-fPIC", "-shared", "-fopenmp", SRC, "-o", out + ".tmp", "-lm"]
    if mutant:
        cmd.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    m = int(sys.argv[1]) if len(sys.argv) > 1 else None
    print(build(m, force=True))
