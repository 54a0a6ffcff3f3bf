"""Compile the fp64 CPU oracle into ``oracle/liboracle.so`` (gcc, OpenMP).

Test infrastructure: the oracle is built so that tests, the smoke check and
the benchmark's CPU-baseline leg can load it. Building it is not using it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pagedkv_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")


def build(source=SOURCE, output=LIBRARY, extra_flags=(), quiet=True):
    """Build the shared library; returns its path. Rebuilds only when stale."""
    if (os.path.exists(output) and not extra_flags
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           *extra_flags, source, "-o", output + ".tmp", "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    if not quiet and res.stderr:
        sys.stderr.write(res.stderr)
    os.replace(output + ".tmp", output)
    return output


if __name__ == "__main__":
    print(build(quiet=False))
