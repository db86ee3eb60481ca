"""Build libmoeffn.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` compiles to its own object in parallel, then nvcc links
them with the static CUDA runtime.  The library takes the driver's TMA
tensor-map encoder through ``cudaGetDriverEntryPointByVersion`` at run time,
so it does not link libcuda and loads on a machine without a GPU driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmoeffn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__])


def up_to_date(lib=LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


# Opt-in instrumented variant: the fused decode kernel records per-CTA clock
# stamps (read back with moe_ffn_debug_fused_timeline), built apart from the
# library the tests and the benchmark load.
TIMELINE_FLAGS = ("-DMOE_FUSED_TIMELINE",)
TIMELINE_BUILD = os.path.join(PKG, "_build_timeline")


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_dir: str = BUILD) -> str:
    """Compile every csrc/*.cu and link libmoeffn.so into out_dir; returns its path."""
    lib = os.path.join(out_dir, "libmoeffn.so")
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_timeline(force: bool = False) -> str:
    """The instrumented variant (see TIMELINE_FLAGS); returns its path."""
    return build(force=force, extra_flags=TIMELINE_FLAGS, out_dir=TIMELINE_BUILD)


if __name__ == "__main__":
    import sys
    if "--timeline" in sys.argv:
        print(build_timeline(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose=True))
