"""Builds the CUDA library libmoe_gb300.so (sm_103a) in-tree under _build/.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library against the shared CUDA runtime.  Run `python -m
moe_expert_layer_03_gb300.build` or call build().
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmoe_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _fingerprint(sources: list[str], extra: list[str]) -> str:
    h = hashlib.sha256()
    for f in sorted(sources + glob.glob(os.path.join(CSRC, "*.cuh")) +
                    [os.path.join(ROOT, "include", "moe.h")]):
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, extra_flags: list[str] | None = None, verbose: bool = False) -> str:
    extra = list(extra_flags or [])
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "fingerprint")
    fp = _fingerprint(sources, extra)
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == fp:
        return LIB
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources))
    tmp = LIB + f".tmp{os.getpid()}"
    # shared CUDA runtime: the library then uses the same runtime instance (current
    # device, streams, events) as the host process's PyTorch
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
                        "-Xlinker", "-rpath,/usr/local/cuda/lib64"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(fp)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
