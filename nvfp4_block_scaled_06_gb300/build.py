"""Build libnvfp4.so in-tree with nvcc for sm_103a (the only target).

Each translation unit compiles in parallel; the shared library links the CUDA
runtime statically, so loading it needs no libcudart on the search path.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libnvfp4.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "gemm_pair.cu", "gemm_skinny.cu", "gemv.cu", "route.cu",
           "static_scratch.cu", "dequant.cu"]
HEADERS = ["ptx.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libnvfp4")
    return cand


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_verbose: bool = False, jobs: int = 8,
          defines=(), lib_path: str | None = None, build_dir: str | None = None) -> str:
    """Compile (if stale) and return the path of libnvfp4.so.

    ``defines`` adds -D flags (e.g. NVFP4_WAIT_STATS for the wait-statistics
    build); such variants go to their own ``lib_path`` / ``build_dir``."""
    lib_out = lib_path or LIB
    bdir = build_dir or BUILD
    os.makedirs(bdir, exist_ok=True)
    dflags = [f"-D{d}" for d in defines]
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "nvfp4.h")]
    cc = nvcc()

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        if _stale(o, [s] + hdrs):
            cmd = [cc, *ARCH, *FLAGS, *dflags, "-c", s, "-o", o]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose or ptxas_verbose:
                print(r.stdout + r.stderr)
        return o

    with ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if _stale(lib_out, objs):
        cmd = [cc, *ARCH, "-shared", "-o", lib_out, *objs, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib_out


LIB_CHECKED = os.path.join(HERE, "libnvfp4_checked.so")


def build_checked(verbose: bool = False) -> str:
    """The build with device-side index checks (NVFP4_CHECKED): violations are
    recorded in the status word as NVFP4_ERR_DEVICE_BOUNDS and the access is
    skipped.  Loaded instead of libnvfp4.so when NVFP4_CHECKED=1."""
    return build(verbose=verbose, defines=("NVFP4_CHECKED",), lib_path=LIB_CHECKED,
                 build_dir=BUILD + "_checked")


if __name__ == "__main__":  # pragma: no cover
    import sys
    if "--checked" in sys.argv:
        print(build_checked(verbose=True))
    else:
        print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
