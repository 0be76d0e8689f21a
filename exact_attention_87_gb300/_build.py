"""Build the sm_103a CUDA library in-tree with nvcc (no cmake, no torch extension).

Each .cu file is compiled to an object in parallel, then linked into
``libfa_gb300.so`` next to this file. The CUDA runtime is linked statically,
so the library needs only the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
SOURCES = ["fa_api.cu", "fa_fwd_f16.cu", "fa_fwd_f32.cu", "fa_fwd_d256.cu", "fa_bwd_f16.cu", "fa_bwd_d256.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-diag-suppress", "1160",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return files


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


TESTING_LIB_PATH = os.path.join(HERE, "libfa_gb300_testing.so")
STRICT_LIB_PATH = os.path.join(HERE, "libfa_gb300_strict.so")


def build(force: bool = False, verbose: bool = False, extra_flags=None, testing: bool = False,
          strict: bool = False) -> str:
    """Build the product library; with testing=True the instrumented testing
    library (-DFA_TESTING: stats/timeline traces and fault injection); with
    strict=True a variant that waits for each P.V to complete before the next
    S = Q K^T reuses its tensor-memory columns (-DFA_STRICT_MMA_ORDER), used by
    the tests to check the default issue order bit for bit."""
    lib_path = TESTING_LIB_PATH if testing else STRICT_LIB_PATH if strict else LIB_PATH
    if not force and up_to_date(lib_path):
        return lib_path
    cc = nvcc()
    objdir = os.path.join(HERE, "_build_testing" if testing else "_build_strict" if strict else "_build")
    os.makedirs(objdir, exist_ok=True)
    extra = list(extra_flags or []) + (["-DFA_TESTING"] if testing else []) + \
        (["-DFA_STRICT_MMA_ORDER"] if strict else [])

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib_path + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, testing="--testing" in sys.argv))
