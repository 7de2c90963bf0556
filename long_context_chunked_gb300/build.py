"""Build the in-tree CUDA library ``libcpattn.so`` for sm_103a with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libcpattn.so")
# Race-detection build: MMA groups serialised (see CPATTN_SERIALIZE_MMA).
LIB_SERIALIZED = os.path.join(PKG, "libcpattn_serialized.so")
# Barrier-count build: every mbarrier arrival and wait counted (see
# CPATTN_COUNT_BARRIERS and cpattn_set_barrier_counts).
LIB_COUNTED = os.path.join(PKG, "libcpattn_counted.so")
VARIANTS = {"release": (LIB, []), "serialized": (LIB_SERIALIZED, ["-DCPATTN_SERIALIZE_MMA"]),
            "counted": (LIB_COUNTED, ["-DCPATTN_COUNT_BARRIERS"])}
SOURCES = ["cpattn.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "cpattn.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build_all(force: bool = False) -> None:
    """Every variant, compiled concurrently."""
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(len(VARIANTS)) as ex:
        for f in [ex.submit(build, force, False, v) for v in VARIANTS]:
            f.result()


def build(force: bool = False, verbose: bool = False, variant: str = "release") -> str:
    lib, defines = VARIANTS[variant]
    if not force and not _stale(lib):
        return lib
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I" + INCLUDE, "-o", lib + ".tmp"] + defines + [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        cmd.insert(2, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    variant = next((v for v in VARIANTS if "--" + v in sys.argv), "release")
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, variant=variant))
