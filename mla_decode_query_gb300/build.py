"""Build ``libmlaqp.so`` in-tree for sm_103a with nvcc (no CMake, no JIT).

``python -m mla_decode_query_gb300.build`` or ``build_library()``.  Each
``.cu`` unit compiles in parallel to an object under ``_build/``; the objects
link into ``mla_decode_query_gb300/_lib/libmlaqp.so`` (CUDA runtime linked
statically, so the library depends only on the driver).  A rebuild happens
when a source or header is newer than the library, or when forced.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG_DIR = Path(__file__).resolve().parent
REPO_DIR = PKG_DIR.parent
CSRC = PKG_DIR / "csrc"
INCLUDE = REPO_DIR / "include"
BUILD_DIR = PKG_DIR / "_build"
LIB_DIR = PKG_DIR / "_lib"
LIB_PATH = LIB_DIR / "libmlaqp.so"

SOURCES = ["mlaqp_api.cu", "mlaqp_kernels_bf16.cu", "mlaqp_kernels_mxfp8.cu", "mlaqp_kernels_large.cu",
           "mlaqp_kernels_v_up.cu", "mlaqp_kernels_warp_bf16.cu", "mlaqp_kernels_warp_mxfp8.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmlaqp.so")


def _inputs() -> list[Path]:
    files = [CSRC / s for s in SOURCES]
    files += list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))
    return files + [Path(__file__)]


def is_stale() -> bool:
    if not LIB_PATH.exists():
        return True
    t = LIB_PATH.stat().st_mtime
    return any(f.stat().st_mtime > t for f in _inputs())


def _compile(src: str, extra: list[str], verbose: bool) -> Path:
    obj = BUILD_DIR / (Path(src).stem + ".o")
    cmd = [nvcc_path(), *ARCH_FLAGS, *COMMON_FLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}")
    return obj


def build_library(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> Path:
    """Compile and link libmlaqp.so if needed; return its path."""
    if not force and not is_stale():
        return LIB_PATH
    BUILD_DIR.mkdir(exist_ok=True)
    LIB_DIR.mkdir(exist_ok=True)
    extra = list(extra_flags or [])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose), SOURCES))
    tmp = LIB_PATH.with_suffix(".so.tmp")
    cmd = [nvcc_path(), *ARCH_FLAGS, "-shared", "-o", str(tmp), *map(str, objs)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError("linking libmlaqp.so failed")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    v = "-v" in sys.argv
    ptx = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build_library(force=True, verbose=v or bool(ptx), extra_flags=ptx))
