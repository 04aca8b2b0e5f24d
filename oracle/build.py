"""Build the CPU oracle (test infrastructure) in place with g++."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def build(force=False):
    src = os.path.join(HERE, "msa_oracle.cpp")
    out = os.path.join(HERE, "liboracle.so")
    if force or not os.path.exists(out) or os.path.getmtime(src) > os.path.getmtime(out):
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-Wall", "-o", out, src])
    return out


if __name__ == "__main__":
    print(build(force=True))
