"""Build step for the CPU oracle library (test infrastructure only).

Compiles ``pa_oracle.c`` with gcc into ``libpa_oracle.so`` beside it.  OpenMP
is used when the compiler supports it; otherwise the oracle runs on one thread.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
LIB = os.path.join(HERE, "libpa_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-o", LIB + ".tmp", SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True, text=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
