"""Builds libbws.so (the CUDA kernels and the C ABI) in this directory.

nvcc compiles every translation unit for sm_103a in parallel, then links one
shared library. No CMake, no torch extension machinery: the library exports
plain C symbols (include/bws.h) and is loaded with ctypes.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbws.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _flags():
    """nvcc flags of every translation unit; BWS_NVCC_FLAGS adds to them (read
    at each build, e.g. -DBWS_TRACE for the opt-in timestamp trace)."""
    return (["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
             "-I", os.path.join(ROOT, "include")] + os.environ.get("BWS_NVCC_FLAGS", "").split())


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbws.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False, force=False):
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    # objects built with other flags (e.g. the opt-in -DBWS_TRACE) are rebuilt
    stamp = os.path.join(BUILD, "flags.txt")
    FLAGS = _flags()
    flags = " ".join(ARCH + FLAGS)
    if not os.path.exists(stamp) or open(stamp).read() != flags:
        force = True
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "bws.h"))
    objs, jobs = [], []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            jobs.append([nvcc] + ARCH + FLAGS + ["-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"])
        os.replace(tmp, LIB)
        with open(stamp, "w") as f:
            f.write(flags)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
