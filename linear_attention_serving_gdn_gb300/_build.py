"""Build libgdn.so in-tree with nvcc for sm_103a (GB300).

Every .cu file under csrc/ is one translation unit, compiled in parallel,
then linked into ``_lib/libgdn.so`` with the static CUDA runtime.  Only
host-portable flags are used, so the same command builds on x86-64 and on
the aarch64 hosts of GB300 machines.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
# GDN_LIB_DIR / GDN_NVCC_EXTRA: alternative output directory and extra nvcc
# flags (e.g. -DGDN_DEBUG_CHECKS for a self-checking build).
OUT_DIR = os.environ.get("GDN_LIB_DIR") or os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libgdn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "gdn.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    tool = os.path.join(OUT_DIR, "gdn_host_cost")
    tool_src = os.path.join(CSRC, "tools", "host_cost.cpp")
    if not os.path.exists(tool) or os.path.getmtime(tool) < max(os.path.getmtime(tool_src), t):
        return False
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "--expt-relaxed-constexpr"]
    common += os.environ.get("GDN_NVCC_EXTRA", "").split()
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [cc, *common, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    build_tools()
    return LIB


HOST_COST = os.path.join(OUT_DIR, "gdn_host_cost")


def build_tools() -> str:
    """Build the host-cost probe (csrc/tools/host_cost.cpp) against the library."""
    src = os.path.join(CSRC, "tools", "host_cost.cpp")
    out = os.path.join(OUT_DIR, "gdn_host_cost")
    cmd = [nvcc(), *ARCH, "-O2", "-std=c++17", "-I", INCLUDE, src, "-o", out, "-L", OUT_DIR, "-lgdn",
           "-Xlinker", "-rpath", "-Xlinker", OUT_DIR, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"host-cost probe build failed:\n{r.stdout}\n{r.stderr}")
    return out


def build_variant(name: str, defines: list[str], force: bool = False) -> str:
    """Build the library with extra preprocessor definitions into
    ``_lib_<name>/libgdn.so`` (used by tests that need a differently
    configured kernel, e.g. a short handshake wait limit)."""
    global OUT_DIR, LIB
    saved = OUT_DIR, LIB, os.environ.get("GDN_NVCC_EXTRA")
    try:
        OUT_DIR = os.path.join(HERE, f"_lib_{name}")
        LIB = os.path.join(OUT_DIR, "libgdn.so")
        os.environ["GDN_NVCC_EXTRA"] = " ".join([saved[2] or ""] + [f"-D{d}" for d in defines]).strip()
        return build(force=force)
    finally:
        OUT_DIR, LIB = saved[0], saved[1]
        if saved[2] is None:
            os.environ.pop("GDN_NVCC_EXTRA", None)
        else:
            os.environ["GDN_NVCC_EXTRA"] = saved[2]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
