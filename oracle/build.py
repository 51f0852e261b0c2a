"""Compile the CPU oracle (plain C, binary64) into oracle/_build/libnvfp4_oracle.so.

Test infrastructure: the library this builds is loaded only by the tests, the
smoke check and the bench's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libnvfp4_oracle.so")


def compile_source(src: str, out: str) -> str:
    """Compile one C file into a shared library (OpenMP when the compiler has it)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)  # no OpenMP runtime: sequential oracle
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_source(SRC, LIB)


if __name__ == "__main__":
    print(build(force=True))
