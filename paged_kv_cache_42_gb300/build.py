"""Build ``libpagedattn.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` file (kernels) is compiled with nvcc and each ``csrc/*.cpp``
file (the host runtime: block pool, block hash, scheduler) with the host C++
compiler, in parallel, then all objects are linked into one shared library with the CUDA runtime linked statically, so the library
has no dependency beyond the driver. Run ``python -m
paged_kv_cache_42_gb300.build`` or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libpagedattn.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


HOST_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-I", CSRC]


def cxx() -> str:
    return os.environ.get("CXX") or shutil.which("g++") or "c++"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


STAMP = os.path.join(BUILD_DIR, "flags.txt")


def extra_flags() -> list:
    """Extra nvcc flags from PA_NVCC_EXTRA (e.g. tuning macros); recorded in a
    stamp so a change of flags triggers a rebuild."""
    return os.environ.get("PA_NVCC_EXTRA", "").split()


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    stamp = open(STAMP).read() if os.path.exists(STAMP) else ""
    if stamp != " ".join(extra_flags()):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
    if src.endswith(".cpp"):
        cmd = [cxx(), *HOST_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"c++ failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra_flags(), "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(STAMP, "w") as f:
        f.write(" ".join(extra_flags()))
    return LIB_PATH


def build_variant(name: str, defines: list) -> str:
    """Build the library with extra preprocessor definitions into its own
    directory and file (``lib<name>.so`` beside the library), leaving the
    library itself untouched. For tests that need a differently configured
    build; the variant is never loaded by the package."""
    out_dir = os.path.join(PKG, "_build_" + name)
    lib = os.path.join(PKG, f"lib{name}.so")
    os.makedirs(out_dir, exist_ok=True)
    flags = [f"-D{d}" for d in defines]

    def one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        if src.endswith(".cpp"):
            cmd = [cxx(), *HOST_FLAGS, "-c", src, "-o", obj]
        else:
            cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build of {name} failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(one, srcs))
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", lib, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {name} failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
