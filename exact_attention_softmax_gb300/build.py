"""Build the C-ABI shared library ``libsdpa_gb300.so`` for sm_103a.

Every ``csrc/*.cu`` translation unit is compiled in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a`` and linked (static CUDA
runtime, no libcuda link: the tensor-map encoder is fetched from the driver
at run time) into ``exact_attention_softmax_gb300/lib/``. Run
``python -m exact_attention_softmax_gb300.build`` or call :func:`build`;
``--debug`` (``build(debug=True)``) builds ``libsdpa_gb300_debug.so`` instead,
compiled with ``SDPA_DEBUG``: device-side bounds checks that skip a refused
access and set a status bit rather than trap. The binding loads it when
``SDPA_GB300_LIB`` names it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libsdpa_gb300.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libsdpa_gb300_debug.so")
# The exponential-unit throughput probe the benchmark measures its ceiling
# with; a library of its own, outside the attention ABI.
PROBE_DIR = os.path.join(PKG, "probe")
PROBE_PATH = os.path.join(LIB_DIR, "libsdpa_probe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(x) > t for x in [src] + _headers())


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile (incrementally) and link the library (``debug``: the build with
    device-side bounds checks); returns its path."""
    nvcc = _nvcc()
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    flags = FLAGS + (["-DSDPA_DEBUG"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    # objects built on another host architecture are never reused
    stamp = os.path.join(build_dir, "HOST_ARCH")
    here = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != here:
        force = True
    srcs = sources()
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(pair):
        src, obj = pair
        if not force and not ptxas_info and not _stale(obj, src):
            return ""
        cmd = [nvcc, *ARCH, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    probe_srcs = sorted(os.path.join(PROBE_DIR, f) for f in os.listdir(PROBE_DIR) if f.endswith(".cu"))

    def build_probe():
        if debug or not force and os.path.exists(PROBE_PATH) and all(
                os.path.getmtime(PROBE_PATH) >= os.path.getmtime(x) for x in probe_srcs):
            return ""
        cmd = [nvcc, *ARCH, *FLAGS, "-shared", "-o", PROBE_PATH, *probe_srcs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for the probe:\n{r.stdout}\n{r.stderr}")
        return ""

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs) + 1)) as ex:
        probe = ex.submit(build_probe)
        logs = list(ex.map(compile_one, zip(srcs, objs)))
        probe.result()
    if verbose or ptxas_info:
        for s, log in zip(srcs, logs):
            if log.strip():
                print(f"== {os.path.basename(s)}\n{log}", file=sys.stderr)
    newest = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(lib_path) or os.path.getmtime(lib_path) < newest:
        tmp = lib_path + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(here + "\n")
    return lib_path


def ensure_built() -> str:
    return build()


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv, force="--force" in sys.argv,
                debug="--debug" in sys.argv))
