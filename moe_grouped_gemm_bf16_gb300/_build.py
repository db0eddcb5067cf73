"""Builds the C-ABI library `libdg.so` (the CUDA kernels and their host
launcher) for sm_103a with nvcc, in the package directory.

`python -m moe_grouped_gemm_bf16_gb300._build` or `build()`.  The translation
units compile in parallel; the result links the CUDA runtime statically so the
library does not depend on which libcudart the process loaded first.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdg.so")
LIB_DEBUG = os.path.join(HERE, "libdg_debug.so")

SOURCES = ["dg_host.cu", "dg_inst_dense.cu", "dg_inst_contiguous.cu", "dg_inst_masked.cu", "dg_inst_mn.cu", "dg_inst_ue8m0.cu", "dg_inst_ue8m0_mn.cu", "dg_inst_bs.cu",
           "dg_inst_bs_mn.cu", "dg_quant.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dg.h")]
    return max(os.path.getmtime(f) for f in files)


def build(force=False, verbose=False, debug=False):
    """Compile the library.  debug=True builds the checked library
    libdg_debug.so instead (every kernel compiled with -DDG_DEBUG=1: bounds
    checks before each TMA load and plain global store, fill checks after
    each ring wait, failures reported in the device status word)."""
    lib = LIB_DEBUG if debug else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps():
        return lib
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE,
             "-I", CSRC]
    if debug:
        flags += ["-DDG_DEBUG=1"]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
