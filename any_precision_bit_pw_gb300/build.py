"""Build libpw.so in-tree for sm_103a (GB300).

    python -m any_precision_bit_pw_gb300.build        # or __graft_entry__.build()

Every translation unit is compiled in parallel with nvcc (CUDA) or g++ (host
C++), then linked into ``any_precision_bit_pw_gb300/libpw.so`` with the CUDA
runtime linked statically.  Objects go to ``_build/`` at the repository root.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpw.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall"]


def _cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _compile(src: str, cuda: str, verbose_ptxas: bool) -> tuple:
    obj = os.path.join(BUILD, src + ".o")
    path = os.path.join(CSRC, src)
    if src.endswith(".cu"):
        cmd = [os.path.join(cuda, "bin", "nvcc"), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC,
               "-c", path, "-o", obj]
        if verbose_ptxas:
            cmd[1:1] = ["-Xptxas", "-v"]
    else:
        cmd = [os.environ.get("CXX", "g++"), *CXX_FLAGS, "-I", INCLUDE, "-I", CSRC,
               "-I", os.path.join(cuda, "include"), "-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr, " ".join(cmd)


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    cuda = _cuda_home()
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda s: _compile(s, cuda, ptxas_info), srcs))
    failed = [r for r in results if r[2] != 0]
    for src, _, rc, out, cmd in results:
        if verbose or rc != 0 or ptxas_info:
            print(f"== {src} (rc={rc})\n{cmd}\n{out}", file=sys.stderr)
    if failed:
        raise RuntimeError("libpw build failed: " + ", ".join(r[0] for r in failed))
    tmp = LIB + ".tmp"
    cmd = [os.path.join(cuda, "bin", "nvcc"), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp,
           *[r[1] for r in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("libpw link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
