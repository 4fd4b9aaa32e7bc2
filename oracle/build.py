"""Builds the CPU oracle shared library (test infrastructure).

The oracle is plain C11 compiled with ``-ffp-contract=off`` so that every
binary32 operation is rounded on its own (no fused multiply-add, which GCC
would otherwise form on aarch64 hosts), and without ``-ffast-math``.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gc_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libgc_oracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing", "-fPIC", "-Wall", "-Wextra",
          "-Wno-maybe-uninitialized"]


def build(force=False):
    """Compiles ``gc_oracle.c`` into ``_build/libgc_oracle.so`` if stale."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-shared", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
