"""Build libkvq.so in-tree: nvcc for sm_103a, one object per translation unit
compiled in parallel, static CUDA runtime, no torch headers.

    python -m paged_quantized_kv_gb300.build [--force] [--ptxas-verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvq.so")

SOURCES = ["kvq_api.cu", "store_nvfp4.cu", "gather_indexer_k.cu",
           "load_nvfp4.cu", "store_indexer_k.cu", "attention_noalloc.cu",
           "paged_attention_mma.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"),
                        "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "kvq.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in _inputs())


def build(force: bool = False, ptxas_verbose: bool = False,
          defines: dict | None = None, out: str | None = None) -> str:
    """Build libkvq.so (or ``out``) if stale; ``defines`` are passed to nvcc
    as -DNAME=VALUE (tuning knobs of the kernels; defaults otherwise)."""
    lib = out or LIB
    if not force and not defines and out is None and not _stale():
        return LIB
    bdir = BUILD if out is None else out + ".build"
    os.makedirs(bdir, exist_ok=True)
    # one build at a time per output (test workers may all ask at once);
    # whoever waited finds the library fresh and returns
    with open(os.path.join(bdir, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and not defines and out is None and not _stale():
            return LIB
        return _build_locked(lib, bdir, ptxas_verbose, defines)


def _build_locked(lib, bdir, ptxas_verbose, defines):
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    extra += [f"-D{k}={v}" for k, v in (defines or {}).items()]

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if ptxas_verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static",
           *[o for o, _ in results], "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv,
                ptxas_verbose="--ptxas-verbose" in sys.argv))
