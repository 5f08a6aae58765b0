"""Compile the C part of the oracle (test infrastructure) with the host gcc.

-ffp-contract=off keeps every multiply and add as written, so the oracle's
arithmetic is the same on x86-64 and aarch64 hosts.
"""
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def build_oracle(verbose: bool = False) -> str:
    src = os.path.join(_HERE, "plmla_oracle.c")
    out = os.path.join(_HERE, "liboracle_plmla.so")
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           src, "-o", tmp, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(verbose=True))
