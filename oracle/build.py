"""Compile the CPU oracle into ``oracle/libmfx_oracle.so``.

TEST INFRASTRUCTURE ONLY: the oracle is loaded by the tests, by the smoke check
and by the CPU-baseline leg of bench.py.  ``-ffp-contract=off`` keeps every
fp32 multiply and add a separate IEEE rounding (gcc would otherwise fuse them on
aarch64); no fast-math flag is given.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mfx_oracle.c")
LIB = os.path.join(HERE, "libmfx_oracle.so")

CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its sources."""
    srcs = [SRC, os.path.join(HERE, "mfx_oracle.h")]
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(s) for s in srcs)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
