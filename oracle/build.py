"""Build the CPU oracle shared libraries (test infrastructure only).

liboracle_f64.so computes in double (the parity truth); liboracle_f32.so in
float, the listing's own precision.  Plain -O2 with OpenMP; no fast-math and no
FMA contraction, so the float build rounds every operation like the listing.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gpt2_oracle.c")
VARIANTS = {"f64": [], "f32": ["-DORACLE_REAL_FLOAT"]}


def lib_path(variant: str) -> str:
    return os.path.join(HERE, f"liboracle_{variant}.so")


def build(force: bool = False) -> None:
    for variant, defs in VARIANTS.items():
        out = lib_path(variant)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
            continue
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-D_DEFAULT_SOURCE", *defs, SRC, "-o", out + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(out + ".tmp", out)


if __name__ == "__main__":
    build(force="--force" in sys.argv)
