"""Build libw4a4.so (and the peak-probe library) in-tree with nvcc for sm_103a.

    python -m hadamard_rotated_w4a4_gb300.build [--probes] [--jobs N]

Each CUDA translation unit is compiled in parallel to an object under
``_build/``; the objects are linked into ``libw4a4.so`` next to this file.
Nothing is installed.  The build is skipped when the library is newer than
every source.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")

LIB_SOURCES = ["act_quant.cu", "pack_weights.cu", "gemm_tc.cu", "gemm_grp.cu", "gemm_id.cu", "gemm_small_m.cu", "capi.cu"]
PROBE_SOURCES = ["probes.cu"]
LIB = os.path.join(PKG, "libw4a4.so")
PROBE_LIB = os.path.join(PKG, "libw4a4_probes.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
           "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the W4A4 CUDA library cannot be built")


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "w4a4.h"))
    return hs


def _stale(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources + _headers())


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, *NVFLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build_lib(target: str, names: list[str], jobs: int, verbose: bool = False, force: bool = False) -> str:
    sources = [os.path.join(CSRC, n) for n in names]
    if not force and not _stale(target, sources):
        return target
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=max(1, jobs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), sources))
    tmp = target + ".tmp"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {target} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, target)
    return target


def build(probes: bool = False, jobs: int | None = None, verbose: bool = False, force: bool = False) -> str:
    jobs = jobs or min(8, os.cpu_count() or 4)
    build_lib(LIB, LIB_SOURCES, jobs, verbose, force)
    if probes:
        build_lib(PROBE_LIB, PROBE_SOURCES, jobs, verbose, force)
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--probes", action="store_true")
    ap.add_argument("--jobs", type=int, default=None)
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    print(build(a.probes, a.jobs, a.verbose, a.force))


if __name__ == "__main__":
    main()
