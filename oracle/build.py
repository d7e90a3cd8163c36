"""Compile the plain-C Q4_0 oracle into a shared library (test infrastructure).

``build(mutant=0)`` writes ``oracle/_build/libq4_0_oracle.so`` (or a mutant
variant used only by the pin-strength tests) with gcc.  The flags keep IEEE
semantics: no fast-math and no FMA contraction, so the fp32 quantizer decision
and the fp64 sums are the ones the C source spells out.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "q4_0_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")

CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-fopenmp", "-std=c11", "-Wall", "-Wextra"]


def lib_path(mutant: int = 0, out_dir: str = None) -> str:
    d = out_dir or BUILD_DIR
    name = "libq4_0_oracle.so" if mutant == 0 else f"libq4_0_oracle_mutant{mutant}.so"
    return os.path.join(d, name)


def build(mutant: int = 0, out_dir: str = None, force: bool = False) -> str:
    """Build (if stale) and return the path of the oracle shared library."""
    out = lib_path(mutant, out_dir)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTANT={int(mutant)}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
