"""Compile the C oracle into ``oracle/liboracle.so`` (test infrastructure).

Plain gcc, OpenMP when the compiler has it, no contraction of multiply-adds so
that the oracle gives the same bits on every host.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def _stale():
    if not os.path.exists(LIB):
        return True
    newest = max(os.path.getmtime(os.path.join(HERE, f))
                 for f in ("oracle.c", "oracle.h"))
    return os.path.getmtime(LIB) < newest


def build(force=False):
    """Build the oracle library if it is missing or older than its sources."""
    if not force and not _stale():
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cc = os.environ.get("CC", "gcc")
    base = [cc] + _FLAGS + [SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the same code, single-threaded.
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
