"""Build step for the C oracle (test infrastructure; see oracle/__init__.py).

Compiles oracle/kda_oracle.c with gcc into oracle/_build/libkda_oracle.so.
Portable C11 (x86_64 and aarch64): no intrinsics, no -march=native, and FP
contraction off so that both machines round the same way.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkda_oracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [
        "gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
        "-ffp-contract=off", "-fno-fast-math", "-D_GNU_SOURCE",
        SRC, "-o", tmp, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
