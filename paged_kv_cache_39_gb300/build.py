"""Build ``libkvpaged.so`` in-tree with nvcc for sm_103a (GB300).

The translation units are compiled in parallel, then linked into one shared
library next to this file.  No cmake, no torch extension machinery: the
library exposes the plain C ABI of ``include/kvpaged.h``.
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
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libkvpaged.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def library_path() -> str:
    return os.path.join(HERE, LIB_NAME)


def nvcc_path() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libkvpaged")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, ptxas_info: bool = False, host_flags=(), out: str = None,
          build_dir: str = None) -> str:
    """Compile every translation unit and link the library.  `host_flags`
    go to the host compiler and linker, one flag each (nvcc splits a flag at
    commas), e.g. sanitizers for a test build; `out` / `build_dir` place such
    a variant away from the product build."""
    nvcc = nvcc_path()
    bdir = build_dir or BUILD_DIR
    os.makedirs(bdir, exist_ok=True)
    host = [x for f in host_flags for x in ("-Xcompiler", f)]
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", *host, "-I", INCLUDE, "-I", CSRC]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose or ptxas_info:
        for obj, log in results:
            if log.strip():
                print(f"== {os.path.basename(obj)}\n{log}")
    out = out or library_path()
    tmp = out + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", *host, "-o", tmp, *[o for o, _ in results], "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
