"""Builds libozemu.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit compiles in parallel to an object under
``_build/<machine>/``; the objects link into ``ozaki_ii_fp64_gb300/_lib/libozemu.so``.
A stamp next to the library records the host machine and the source hashes,
so a library built on another architecture or from older sources is rebuilt.
"""

import hashlib
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIBNAME = "libozemu.so"
SOURCES = ["api.cu", "split.cu", "gemm_fp4.cu", "crt.cu", "igemm_mma.cu", "gemv.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def lib_path():
    return os.path.join(LIBDIR, LIBNAME)


def _fingerprint():
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode())
                    h.update(f.read())
    h.update(" ".join(ARCH_FLAGS).encode())
    return h.hexdigest()


def _stamp_path():
    return lib_path() + ".stamp"


def is_current():
    if not os.path.exists(lib_path()) or not os.path.exists(_stamp_path()):
        return False
    with open(_stamp_path()) as f:
        return f.read().strip() == _fingerprint()


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link libozemu.so; returns its path."""
    if not force and is_current():
        return lib_path()
    obj_dir = os.path.join(ROOT, "_build", platform.machine())
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    common = ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                           "--expt-relaxed-constexpr"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, res.stdout, res.stderr))
        if verbose or ptxas_info:
            print(res.stdout + res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path() + ".tmp"
    cmd = [cc] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs + ["-lcuda"] * 0
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (res.stdout, res.stderr))
    os.replace(tmp, lib_path())
    with open(_stamp_path(), "w") as f:
        f.write(_fingerprint())
    return lib_path()


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
