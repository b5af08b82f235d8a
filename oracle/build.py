"""Compile the CPU oracle (test infrastructure) into oracle/_build/liboracle.so.

Plain g++ with OpenMP when the compiler has it; no CUDA is involved.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "xmod_oracle.cpp"), os.path.join(HERE, "xmod_oracle_bwd.cpp")]
OUT_DIR = os.path.join(HERE, "_build")
OUT = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(OUT) and all(
            os.path.getmtime(OUT) >= os.path.getmtime(s) for s in SRCS):
        return OUT
    base = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", *SRCS, "-o", OUT + ".tmp"]
    try:
        subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(OUT + ".tmp", OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
