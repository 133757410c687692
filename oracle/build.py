"""Compile the CPU oracle (plain C, gcc) into ``oracle/liboracle.so``.

Test infrastructure: the oracle is built alongside the CUDA library so the
tests, the smoke check and the benchmark's CPU-baseline leg can load it; the
product path never does.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

# -ffp-contract=off: no fused multiply-adds; every fp32 operation rounds once
# as written.  No -ffast-math, no -march=native (the library must build and
# give the same results on x86-64 and aarch64).
_BASE = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
         "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                               os.path.getmtime(SRC[:-1] + "h"))):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = _BASE + ["-fopenmp", "-o", tmp, SRC, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        # No OpenMP runtime: the pragmas are ignored and the oracle runs on
        # one thread.
        cmd = _BASE + ["-o", tmp, SRC, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
