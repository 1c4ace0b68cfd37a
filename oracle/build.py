"""Compile the CPU oracle (plain C) into a shared library.

Test infrastructure: the oracle is only built and loaded by the test suite,
the smoke check and the benchmark's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_SO = os.path.join(HERE, "liboracle.so")

# -ffp-contract=off: every fp32 operation in oracle.c is rounded on its own
# (gcc contracts a*b+c into an fma by default on aarch64).  No -ffast-math.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def build(src=None, out=None, quiet=True):
    """Compile ``src`` (default: oracle/oracle.c) into ``out``; return ``out``."""
    src = src or os.path.join(HERE, "oracle.c")
    out = out or DEFAULT_SO
    tmp = f"{out}.tmp{os.getpid()}"      # one file per process, renamed over the old
    cmd = ["gcc", *CFLAGS, "-I", HERE, src, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        if os.path.exists(tmp):
            os.remove(tmp)
        raise RuntimeError("oracle build failed:\n" + res.stderr)
    if not quiet and res.stderr:
        print(res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(quiet=False))
