"""Builds the CPU oracle library (test infrastructure only).

`python -m oracle.build` (or `build()` from `__graft_entry__`) compiles
`ref_gemm.c` with gcc into `libdgref.so` beside it.  `build_mutant(n)` compiles
a copy with one deliberate mistake (`-DDG_REF_MUTANT=n`) into a temporary
directory, for the tests that show the pins catch such mistakes.
"""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ref_gemm.c")
LIB = os.path.join(HERE, "libdgref.so")


def _compile(out, defines=()):
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-std=c11", SRC,
           "-o", out, "-lm"]
    cmd[1:1] = [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    return out


def build(force=False):
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        _compile(tmp)
        os.replace(tmp, LIB)
    return LIB


def build_mutant(n, outdir=None):
    outdir = outdir or tempfile.mkdtemp(prefix="dgref_mut")
    return _compile(os.path.join(outdir, f"libdgref_mut{n}.so"), [f"DG_REF_MUTANT={n}"])


if __name__ == "__main__":
    print(build(force=True))
