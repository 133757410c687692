"""Build the CUDA library ``lib/libmoe_gb300.so`` in-tree with nvcc.

sm_103a only (GB300).  The translation units compile in parallel; the host
runtime links the CUDA runtime statically, so the library needs nothing but
the CUDA driver (libcuda) at load time.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmoe_gb300.so")
SOURCES = ["gemm.cu", "gemm_pair.cu", "decode.cu", "route.cu", "prep.cu", "api.cu",
           "route_static.cu", "peak.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                    if f.endswith((".cuh", ".h"))] + [os.path.join(ROOT, "include", "moe.h")]
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False):
    os.makedirs(os.path.join(LIBDIR, "obj"), exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(LIBDIR, "obj", s + ".o")
        if force or _stale(obj, src):
            jobs.append([nvcc] + _flags() + ["-c", src, "-o", obj])
    errors = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, r in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
            if r.returncode != 0:
                errors.append(" ".join(cmd) + "\n" + r.stderr)
            elif verbose and r.stderr:
                print(r.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    objs = [os.path.join(LIBDIR, "obj", s + ".o") for s in SOURCES]
    if force or jobs or not os.path.exists(LIB):
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
