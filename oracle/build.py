"""Build the C oracle (``liboracle.so``) with the host compiler.

Test infrastructure only: the product library never links or loads it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "msm_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, out: str = None, mutation: int = 0) -> str:
    """Compile msm_oracle.c into a shared library and return its path.

    ``mutation`` > 0 builds a variant with one planted mistake (see the
    ORACLE_MUTATION switch in msm_oracle.c); it must go to a separate ``out``.
    """
    out = out or LIB
    if mutation and out == LIB:
        raise ValueError("a mutated oracle must not replace liboracle.so")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O3", "-std=gnu11", "-fPIC", "-shared", "-pthread",
           "-DORACLE_MUTATION=%d" % mutation, SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
