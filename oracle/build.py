"""Compile the CPU oracle (test infrastructure) into oracle/_build/libdt_oracle.so.

Plain gcc, no vendor toolchain.  -ffp-contract=off keeps every fp32 multiply and
add separately rounded on both x86-64 and aarch64 (gcc contracts a*b+c into an
fma by default on aarch64), so the oracle's fp32 decisions are reproducible.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dt_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libdt_oracle.so")

CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard", "-Wall"]


def compile_to(src: str, out: str) -> str:
    """Compile an oracle source file into the shared library `out` (same flags)."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle if its library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    return compile_to(SRC, LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
