"""Builds libmoe_w4.so in-tree with nvcc for sm_103a (translation units
compiled in parallel, then linked).  Run as `python -m bit_quantized_sparse_gb300._build`.

`--debug` (build(debug=True)) builds libmoe_w4_debug.so instead: the same
sources with MW4_DEBUG_CHECKS defined, which adds device-side bounds checks on
every index the kernels read from the routing records (positions, block
records, units); a failed check sets MOE_W4_STATUS_BAD_INDEX in the status
word and the access is clamped into range instead of made.  The binding loads
it when the environment has MOE_W4_DEBUG=1."""
import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_w4.so")
LIB_DEBUG = os.path.join(PKG, "libmoe_w4_debug.so")
SOURCES = ["api.cu", "router.cu", "grouping.cu", "decode.cu", "grouped_gemm.cu", "noalloc.cu", "decode_fused.cu",
           "ablation.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _newer(out, deps):
    return os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(d) for d in deps)


def build(verbose=False, force=False, debug=False):
    nvcc = _nvcc()
    bdir, lib = (os.path.join(BUILD, "debug"), LIB_DEBUG) if debug else (BUILD, LIB)
    flags = FLAGS + (["-DMW4_DEBUG_CHECKS"] if debug else [])
    os.makedirs(bdir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "moe_w4.h"))
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or not _newer(o, [s] + headers):
            jobs.append([nvcc] + ARCH + flags + ["-c", s, "-o", o])
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
            if verbose or res.returncode:
                sys.stderr.write(res.stdout + res.stderr)
            if res.returncode:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or not _newer(lib, objs):
        cmd = [nvcc] + ARCH + ["-shared", "-o", lib] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("link failed")
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
