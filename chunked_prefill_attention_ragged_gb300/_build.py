"""In-tree build of libmla_prefill.so with nvcc for sm_103a.

Objects go to ``_build/`` at the repository root; the shared library lands
next to this file.  A stamp (source hash + flags + host machine) decides
whether a rebuild is needed, so importing after a build costs nothing.
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
BUILD_DIR = os.path.join(REPO_DIR, "_build")
LIB_NAME = "libmla_prefill.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

SOURCES = [
    "mla_abi.cpp",
    "planner.cpp",
    "tma.cpp",
    "attn_kernel.cu",
    "gather_kernel.cu",
    "cache_write_kernel.cu",
    "merge_kernel.cu",
    "up_proj_kernel.cu",
    "noalloc.cu",
    "fp8_gather_kernel.cu",
    "absorbed_kernel.cu",
]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmla_prefill.so")


def _stamp() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    h.update(" ".join(ARCH_FLAGS + COMMON_FLAGS).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def _stamp_path() -> str:
    return os.path.join(BUILD_DIR, "stamp.txt")


def is_current() -> bool:
    if not os.path.exists(LIB_PATH) or not os.path.exists(_stamp_path()):
        return False
    with open(_stamp_path()) as f:
        return f.read().strip() == _stamp()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every translation unit (in parallel) and link the shared library."""
    if not force and is_current():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [nvcc, *ARCH_FLAGS, *COMMON_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(_stamp_path(), "w") as f:
        f.write(_stamp())
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
