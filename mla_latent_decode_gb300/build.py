"""Build the CUDA library libmla_decode.so in-tree (nvcc, sm_103a only).

Each translation unit compiles in its own nvcc process, in parallel, then
nvcc links them into one shared library that depends only on the C/C++
runtime (cudart is linked statically; the driver's tensor-map encoder is
looked up at run time), so the library also loads on a machine without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmla_decode.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def _deps_mtime():
    return max(os.path.getmtime(os.path.join(CSRC, f)) for f in os.listdir(CSRC))


def _compile(src: str, log: list) -> str:
    obj = os.path.join(OBJ, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-I", os.path.join(HERE, "..", "include"),
           "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log.append((src, r.stdout + r.stderr))
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/ into libmla_decode.so next to this file; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
            _deps_mtime(), os.path.getmtime(os.path.join(HERE, "..", "include",
                                                         "mla_decode.h"))):
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    log: list = []
    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, log), srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    with open(os.path.join(OBJ, "ptxas.log"), "w") as f:
        for src, out in log:
            f.write(f"== {os.path.basename(src)}\n{out}\n")
    if verbose:
        print(open(os.path.join(OBJ, "ptxas.log")).read(), file=sys.stderr)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
