"""Builds the CUDA library libpi_attn.so for sm_103a with nvcc (no cmake).

Translation units are compiled in parallel into ``_build/`` and linked into
``_lib/libpi_attn.so`` inside the package, next to the Python binding.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libpi_attn.so")

SOURCES = ["api.cu", "pi_simt.cu", "pi_fwd_tc.cu", "pi_bwd_tc.cu", "pi_decode.cu"]
HEADERS = ["pi_common.cuh", "pi_launch.h", "pi_tc_ptx.cuh"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    for cand in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(nv)), "lib64")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library.  Extra nvcc flags (e.g. -D tuning macros) can be given
    in the PI_ATTN_NVCC_EXTRA environment variable; a change of them forces a rebuild."""
    nv = nvcc()
    extra = os.environ.get("PI_ATTN_NVCC_EXTRA", "").split()
    stamp = os.path.join(BUILD_DIR, "extra_flags.txt")
    os.makedirs(BUILD_DIR, exist_ok=True)
    prev = open(stamp).read() if os.path.exists(stamp) else ""
    if prev != " ".join(extra):
        force = True
        with open(stamp, "w") as fh:
            fh.write(" ".join(extra))
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "pi_attn.h")]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or ptxas_info or _stale(o, [s] + headers):
            cmd = [nv, "-c", s, "-o", o] + ARCH_FLAGS + NVCC_FLAGS + extra
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_info or r.returncode != 0:
                    sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed for {cmd[2]}")
    if force or jobs or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nv, "-shared", "-o", tmp] + objs + ARCH_FLAGS + [
            "-cudart", "shared", "-Xlinker", "-rpath," + _cuda_lib_dir(nv)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("link of libpi_attn.so failed")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
