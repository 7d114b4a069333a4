"""Build libcarat.so in-tree with nvcc for sm_103a (GB300).

Each .cu file is compiled to an object in parallel, then linked into one shared
library next to this file.  No cmake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libcarat.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, *ARCH]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcarat.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "carat.h"))
    if os.path.exists(obj) and all(os.path.getmtime(obj) >= os.path.getmtime(d) for d in deps):
        return obj
    cmd = [nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as pool:
        objs = list(pool.map(lambda s: _compile(s, verbose), srcs))
    if os.path.exists(LIBRARY) and all(os.path.getmtime(LIBRARY) >= os.path.getmtime(o)
                                       for o in objs):
        return LIBRARY
    tmp = LIBRARY + ".tmp"
    cmd = [nvcc(), "-shared", *ARCH, "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath", "-Xlinker", "/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


PROBE_SOURCE = os.path.join(os.path.dirname(HERE), "tests", "cuda", "tc_probe.cu")
PROBE_LIBRARY = os.path.join(os.path.dirname(HERE), "tests", "cuda", "_build", "libtc_probe.so")


def build_probe() -> str:
    """Test-only library that checks the tensor-core primitives on a GPU."""
    if not os.path.exists(PROBE_SOURCE):
        return ""
    os.makedirs(os.path.dirname(PROBE_LIBRARY), exist_ok=True)
    deps = [PROBE_SOURCE] + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                             if f.endswith((".cuh", ".h"))]
    if os.path.exists(PROBE_LIBRARY) and all(os.path.getmtime(PROBE_LIBRARY) >= os.path.getmtime(d)
                                             for d in deps):
        return PROBE_LIBRARY
    cmd = [nvcc(), *NVCC_FLAGS, "-shared", "-cudart", "shared", "-o", PROBE_LIBRARY,
           PROBE_SOURCE, "-Xlinker", "-rpath", "-Xlinker", "/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for the probe:\n{r.stdout}\n{r.stderr}")
    return PROBE_LIBRARY


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
