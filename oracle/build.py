"""Compile the fp64 CPU oracle (test infrastructure) into oracle/libqmoe_oracle.so.

Plain C11 with floating-point contraction off, so the oracle's double
arithmetic is the same on x86-64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qmoe_oracle.c")
LIB = os.path.join(HERE, "libqmoe_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           SRC, "-o", LIB + ".tmp", "-lm"]
    subprocess.check_call(cmd)
    os.replace(LIB + ".tmp", LIB)
    return LIB


def build_variant(plant: int, out_path: str) -> str:
    """A deliberately wrong oracle (ORACLE_PLANT=plant) for the pin tests."""
    cmd = ["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
           "-DORACLE_PLANT=%d" % plant, SRC, "-o", out_path, "-lm"]
    subprocess.check_call(cmd)
    return out_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
