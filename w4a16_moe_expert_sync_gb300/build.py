"""Build libw4moe.so in-tree with nvcc for sm_103a (one -gencode, parallel TUs)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libw4moe.so")
SOURCES = ["api.cu", "quantize.cu", "route_align.cu", "combine.cu", "grouped_gemm.cu",
           "static_scratch.cu", "rmsnorm.cu", "sampler.cu", "dense_gemm.cu"]
HEADERS = ["launch.h", "ptx.cuh", "korder.cuh", "combine_fold.cuh", "checks.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(ROOT, "include", "w4moe.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every translation unit and link the shared library; returns its path."""
    if not force and not ptxas_info and not _stale():
        return LIB
    return _compile(BUILD, LIB, [], verbose, ptxas_info)


def build_checked(out_dir: str) -> str:
    """The library with W4_CHECK_BOUNDS (every data-dependent global store
    range-checked; a failed check sets W4_DEV_OUT_OF_BOUNDS and skips the
    store), built into out_dir for the tests; returns its path."""
    return _compile(out_dir, os.path.join(out_dir, "libw4moe_checked.so"), ["-DW4_CHECK_BOUNDS"],
                    False, False)


def _compile(build_dir: str, lib: str, defines: list, verbose: bool, ptxas_info: bool) -> str:
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr", *defines]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))
