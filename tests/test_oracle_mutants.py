"""Mutation sweep over the oracle: the pages' nine mutations, each must turn the pins red.

The mutation list is the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)", section
"Evidence", mutation table (M1..M9), kept with that page's protocol:
  * a pristine control run goes first, under the identical command and filter, and
    must pass (a filter that selects nothing would otherwise score a false catch);
  * a mutant that fails to build is not a catch (the build is -Wall -Wextra -Werror and
    must succeed; every mutant keeps its variables read);
  * the verdict is the child's exit code, never its printed summary line.
Mutations are planted in the oracle only, on the CPU; each build is a separate shared
library selected through SSD_ORACLE_LIB.
"""
import os
import subprocess
import sys

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

MUTANTS = {
    1: ("drop the inter-chunk state term", "chunk_size_invariance"),
    2: ("ignore initial_states", "bruteforce or split_sequence or closed_form"),
    3: ("read states[c] for states[c-1]", "chunk_size_invariance"),
    4: ("drop the D skip connection", "bruteforce or closed_form or decode_continues"),
    5: ("ignore state_indices", "decode_indices or decode_continues"),
    6: ("NULL row as slot 0", "decode_indices"),
    7: ("whole-row variance, not per-group", "norm"),
    8: ("sigmoid instead of silu", "norm"),
    9: ("drop the decode A < 0 check", "decode_rejects or decode_accepts"),
}


def _run(lib, kfilter):
    env = dict(os.environ, SSD_ORACLE_LIB=lib, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider",
           "-k", kfilter]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("k", sorted(MUTANTS))
def test_mutant_is_caught(k):
    what, kfilter = MUTANTS[k]
    pristine = obuild.build()
    rc0, out0 = _run(pristine, kfilter)
    assert rc0 == 0, f"control run under filter {kfilter!r} failed:\n{out0}"
    assert "passed" in out0 and " 0 passed" not in out0, out0
    mutant = obuild.build(mutant=k)           # raises if the mutant does not compile
    rc, out = _run(mutant, kfilter)
    assert rc != 0, f"M{k} ({what}) was NOT caught under filter {kfilter!r}:\n{out}"
    assert rc == 1, f"M{k} ended with exit code {rc}, not a test failure:\n{out}"
