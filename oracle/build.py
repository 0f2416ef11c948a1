"""Compile the fp64 CPU oracle (``oracle.c``) into ``oracle/_lib/liboracle.so``.

Test infrastructure: the oracle is built so that the test suite and the
benchmark's CPU baseline can call it.  Plain ``gcc -O2 -fopenmp``; no
architecture-specific flags, so the same source builds on x86_64 and aarch64.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def command():
    return ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
            "-o", LIB, SRC, "-lm"]


def up_to_date():
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC)


def start():
    """Launch the compile as a subprocess (or return None when up to date)."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if up_to_date():
        return None
    return subprocess.Popen(command(), stdout=subprocess.PIPE, stderr=subprocess.STDOUT)


def build():
    proc = start()
    if proc is None:
        return LIB
    out, _ = proc.communicate()
    if proc.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + out.decode(errors="replace"))
    return LIB


if __name__ == "__main__":
    print(build())
