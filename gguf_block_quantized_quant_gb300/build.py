"""Builds libqg.so in-tree with nvcc for sm_103a (GB300).

The CUDA sources are compiled in parallel: the C-ABI translation unit once, and
``qg_fmt.cu`` once per block format (``-DQG_FMT=<GGUF type id>``).  The library links the
shared CUDA runtime so that it shares the process's runtime state (current device,
streams) with PyTorch.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libqg.so")

FORMATS = {"q4_0": 2, "q4_1": 3, "q5_0": 6, "q5_1": 7, "q8_0": 8, "q2_k": 10, "q3_k": 11, "q4_k": 12, "q5_k": 13,
           "q6_k": 14, "iq4_nl": 20, "iq4_xs": 23}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libqg")
    return p


def _cuda_lib_dir() -> str:
    nv = os.path.realpath(_nvcc())
    return os.path.join(os.path.dirname(os.path.dirname(nv)), "lib64")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(INCLUDE, "qg.h"), __file__])


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC,-O2",
            "-I", CSRC, "-I", INCLUDE, *extra]


def _units():
    units = [(os.path.join(CSRC, "qg_abi.cu"), os.path.join(OUT_DIR, "qg_abi.o"), [])]
    for name, fid in FORMATS.items():
        units.append((os.path.join(CSRC, "qg_fmt.cu"), os.path.join(OUT_DIR, f"qg_fmt_{name}.o"),
                      [f"-DQG_FMT={fid}"]))
    return units


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    """Compile (if needed) and return the path of libqg.so."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(u):
        src, obj, extra = u
        cmd = [nvcc, *_flags(extra), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{r.stderr[-6000:]}")
        if verbose and r.stderr.strip():
            print(r.stderr)
        return obj

    units = _units()
    workers = jobs or min(len(units), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(compile_one, units))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{_cuda_lib_dir()}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libqg.so failed:\n{r.stderr[-6000:]}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
