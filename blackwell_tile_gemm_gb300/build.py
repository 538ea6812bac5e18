"""Builds libtgemm.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

Each translation unit compiles in its own nvcc process, in parallel; the
objects are linked into ``blackwell_tile_gemm_gb300/_build/libtgemm.so``.  The
probe kernels (the pages' worked examples, the tensor-pipe rate probe and the
SM occupier the tests and the benchmark use) go into a separate
``libtgemm_probes.so`` that links against it, so the product library carries
only the contraction's entry points.

    python -m blackwell_tile_gemm_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libtgemm.so")
PROBE_LIB = os.path.join(BUILD, "libtgemm_probes.so")
SOURCES = ["api.cu", "gemm_bf16.cu", "gemm_blockscaled.cu", "gemm_fp4.cu", "gemm_skinny.cu",
           "gemm_gather.cu", "gemm_mxfp8_noalloc.cu", "transpose.cu"]
PROBE_SOURCES = ["probes.cu"]
HEADERS = ["tg_ptx.cuh", "gemm_kernel.cuh", "gemm_launch.cuh", "tg_internal.h", "epilogue.cuh",
           "gemm_kinds.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _inputs_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + PROBE_SOURCES + HEADERS]
    paths += [os.path.join(ROOT, "include", f) for f in ("tgemm.h", "tgemm_probes.h")]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def up_to_date() -> bool:
    t = _inputs_mtime()
    return all(os.path.exists(p) and os.path.getmtime(p) >= t for p in (LIB, PROBE_LIB))


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(os.path.join(BUILD, "obj"), exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, "obj", src.replace(".cu", ".o"))
        cmd = [cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if ptxas_verbose or verbose:
            sys.stderr.write(r.stderr)
        return obj

    all_sources = SOURCES + PROBE_SOURCES
    workers = min(len(all_sources), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = dict(zip(all_sources, ex.map(compile_one, all_sources)))

    def link(out, srcs, extra):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [objs[s] for s in srcs] + extra
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(out)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)

    link(LIB, SOURCES, [])
    # The probes call the library's internal helpers (device context, tensor
    # maps, the status record): link against it, found next to this file.
    link(PROBE_LIB, PROBE_SOURCES, ["-L", BUILD, "-ltgemm", "-Xlinker", "-rpath,$ORIGIN"])
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose))


if __name__ == "__main__":
    main()
