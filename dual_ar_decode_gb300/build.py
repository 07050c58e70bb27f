"""Compile the CUDA library libtf_dualar.so for sm_103a, in-tree.

Each .cu translation unit is compiled in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a), then linked into a shared library
next to this file.  Rebuilds only when a source is newer than the library.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libtf_dualar.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["tf_api.cu", "kernels_gemv.cu", "kernels_attn.cu", "kernels_misc.cu", "kernels_umma.cu"]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tf.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False,
          defines=(), out: str | None = None) -> str:
    """Build the library.  `defines` (e.g. ["TF_GEMV_RING_BYTES=131072"]) and
    `out` build a variant elsewhere, for tuning sweeps."""
    lib_path = out or LIB
    if not force and not ptxas_info and not defines and out is None and up_to_date():
        return LIB
    build_dir = BUILD_DIR if out is None else out + ".objs"
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    extra += [f"-D{d}" for d in defines]

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc(), *NVCC_FLAGS, *extra, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            sys.stderr.write(err)
    objs = [o for o, _ in results]
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs,
           "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, ptxas_info="--ptxas" in sys.argv))
