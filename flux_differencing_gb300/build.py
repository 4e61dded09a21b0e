"""Build the CUDA library libesdg.so in-tree (sm_103a only).

Compiles every translation unit with nvcc in parallel -- the volume kernel
once per (order N, precision) -- and links them with the shared CUDA runtime.
Rebuilds only when a source is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libesdg.so")
# Debug variant: the same sources with -DESDG_DEBUG_CHECKS=1 (every kernel index
# range-checked into ESDG_STATUS_INDEX, shared memory poisoned with NaN before
# use), for the tests only.
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libesdg_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-O2", f"-I{CSRC}", f"-I{INCLUDE}"] + ARCH


def _nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libesdg.so")


def _units():
    units = [("esdg_api", os.path.join(CSRC, "esdg_api.cu"), []),
             ("geometry", os.path.join(CSRC, "geometry.cu"), []),
             ("peak_bench", os.path.join(CSRC, "peak_bench.cu"), []),
             ("esdg_noalloc", os.path.join(CSRC, "esdg_noalloc.cu"), []),
             ("index_check", os.path.join(CSRC, "index_check.cu"), []),
             ("time", os.path.join(CSRC, "time_kernel.cu"), []),
             ("pipeline", os.path.join(CSRC, "esdg_pipeline.cu"), [])]
    for prec, tag in ((0, "fp64"), (1, "fp32"), (2, "fp64ff")):
        units.append((f"surface_{tag}", os.path.join(CSRC, "surface_kernel.cu"), [f"-DESDG_SURF_PREC={prec}"]))
    for n in range(1, 9):
        for prec, tag in ((0, "fp64"), (1, "fp32"), (2, "fp64ff")):
            units.append((f"volume_{tag}_n{n}", os.path.join(CSRC, "volume_inst.cu"),
                          [f"-DESDG_INST_N={n}", f"-DESDG_INST_PREC={prec}"]))
    return units


def _sources():
    out = []
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".cu", ".cuh", ".h", ".inc")):
                out.append(os.path.join(d, f))
    out.append(os.path.abspath(__file__))
    return out


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, jobs: int | None = None,
          debug: bool = False) -> str:
    """Compile and link libesdg.so (or, with debug=True, libesdg_debug.so with the
    kernels' index checks compiled in); returns its path."""
    lib_path, build_dir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and not ptxas_info and not _stale(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DESDG_DEBUG_CHECKS=1"] if debug else [])

    def compile_one(u):
        name, src, defs = u
        obj = os.path.join(build_dir, name + ".o")
        cmd = [nvcc, "-c", src, "-o", obj] + NVCC_FLAGS + defs + extra
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {name}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, (r.stdout + r.stderr)

    units = _units()
    nj = jobs or min(len(units), max(1, os.cpu_count() or 1))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=nj) as ex:
        results = list(ex.map(compile_one, units))
    objs = [r[0] for r in results]
    logs = [r[1] for r in results]
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "shared"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    if verbose or ptxas_info:
        for u, log in zip(units, logs):
            if log.strip():
                sys.stdout.write(f"== {u[0]}\n{log}")
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
