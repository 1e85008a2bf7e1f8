"""Build the kv4 CUDA libraries in-tree for GB300 (sm_103a).

libkv4.so is the decode library (include/kv4.h); libkv4_diag.so holds the
tensor-pipe rate probes (include/kv4_diag.h), which only the benchmark's
report mode loads.  Each translation unit is compiled in parallel with nvcc,
then linked into a shared library against the shared CUDA runtime (the same
libcudart that PyTorch loads).  The results sit next to this file and are
git-ignored.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libkv4.so")
DIAG_OUT = os.path.join(HERE, "libkv4_diag.so")
BUILD_DIR = os.path.join(ROOT, "_build")
SOURCES = ["kv4_abi.cu", "kv4_append.cu", "kv4_decode.cu", "kv4_decode_mma.cu",
           "kv4_decode_stream.cu", "kv4_decode_bf16.cu", "kv4_noalloc.cu"]
DIAG_SOURCES = ["diag/kv4_diag.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the kv4 CUDA library cannot be built")


def _deps():
    files = []
    for d, _, names in os.walk(CSRC):
        files += [os.path.join(d, f) for f in names]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(OUT) or not os.path.exists(DIAG_OUT):
        return True
    t = min(os.path.getmtime(OUT), os.path.getmtime(DIAG_OUT))
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return OUT
    nvcc = _nvcc()
    cuda_home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     f"-I{INCLUDE}", "-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(os.path.splitext(src)[0]) + ".o")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(obj + ".log", "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES) + len(DIAG_SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES + DIAG_SOURCES))
    for out, part in ((OUT, objs[:len(SOURCES)]), (DIAG_OUT, objs[len(SOURCES):])):
        tmp = out + f".{os.getpid()}.tmp"
        link = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + part + [
            "-Xlinker", f"-rpath,{os.path.join(cuda_home, 'lib64')}"]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, out)
        if verbose:
            print(f"built {out}")
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
