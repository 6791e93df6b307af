"""Compile the oracle (plain C, fp64) into ``oracle/libbqoracle.so``.

Test infrastructure only.  gcc flags keep IEEE-754 fp32 semantics exact: no
fast-math and no FMA contraction, so the packer's divisions and roundings are
the ones written in the source on both x86_64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bq_oracle.c")
LIB = os.path.join(HERE, "libbqoracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]


def compile_oracle(src=SRC, out=LIB, force=False):
    """Build ``out`` from ``src`` unless it is newer than the source."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", *CFLAGS, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)  # atomic: concurrent builders never see a half file
    return out


if __name__ == "__main__":
    print(compile_oracle(force="--force" in sys.argv))
