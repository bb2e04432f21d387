"""Build libdsa.so in-tree for sm_103a (GB300).

Each CUDA translation unit compiles in parallel with nvcc, then the objects are
linked into ``_build/libdsa.so`` (cudart linked dynamically, so the library
shares the CUDA runtime PyTorch has already loaded).  A stamp of the sources and
flags skips the build when nothing changed.

    python -m sparse_attention_indexer_kpool_gb300.build
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libdsa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", INCLUDE]
SOURCES = ["dsa_abi.cu", "kpool_compress.cu", "index_scores.cu", "index_scores_umma.cu",
           "topk.cu", "mla_decode.cu", "mla_umma.cu", "select_noalloc.cu",
           "indexer_proj.cu"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libdsa needs the CUDA 13 toolkit to build")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stamp() -> str:
    h = hashlib.sha256()
    h.update(" ".join(NVCC_FLAGS).encode())
    names = sorted(os.listdir(CSRC)) + ["../include/dsa.h"]
    for n in names:
        p = os.path.normpath(os.path.join(CSRC, n))
        if os.path.isfile(p):
            h.update(n.encode())
            h.update(open(p, "rb").read())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile libdsa.so if needed; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp_path = os.path.join(BUILD, "stamp")
    stamp = _stamp()
    if (not force and os.path.exists(LIB) and os.path.exists(stamp_path)
            and open(stamp_path).read() == stamp):
        return LIB
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc] + NVCC_FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        with open(os.path.join(BUILD, src.replace(".cu", ".ptxas.txt")), "w") as f:
            f.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    libdir = _cuda_lib_dir(nvcc)
    tmp = LIB + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-L", libdir, "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    if verbose:
        for src in SOURCES:
            print(open(os.path.join(BUILD, src.replace(".cu", ".ptxas.txt"))).read())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
