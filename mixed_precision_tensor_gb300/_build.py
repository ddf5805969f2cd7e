"""Build libtcg.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each .cu file compiles to an object in parallel; the objects link into
``mixed_precision_tensor_gb300/_lib/libtcg.so`` with a static CUDA runtime.  A stamp
beside the library (``libtcg.so.key``) records a hash of the sources, the flags and the
host architecture; the library is rebuilt whenever that key differs.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(ROOT, "_build", "tcg")
LIB_PATH = os.path.join(OUT_DIR, "libtcg.so")
SOURCES = ["tcg_api.cu", "tcg_kernels.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cand, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC"]


def _deps():
    return sorted([os.path.join(CSRC, f) for f in os.listdir(CSRC)] +
                  [os.path.join(INCLUDE, "tcg.h")])


def source_key(deps=None) -> str:
    """What a build depends on: the sources' contents, the compiler flags and the host
    architecture (a library built on another machine, or from other sources, is stale
    whatever its modification time)."""
    h = hashlib.sha256()
    for d in (deps if deps is not None else _deps()):
        h.update(os.path.basename(d).encode() + b"\0")
        with open(d, "rb") as f:
            h.update(f.read())
    h.update(" ".join(FLAGS).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def stamp_path(lib_path: str) -> str:
    return lib_path + ".key"


def up_to_date(lib_path: str = LIB_PATH, key: str | None = None) -> bool:
    """True when ``lib_path`` exists and its stamp records the current source key."""
    if not os.path.exists(lib_path) or not os.path.exists(stamp_path(lib_path)):
        return False
    with open(stamp_path(lib_path)) as f:
        return f.read().strip() == (key if key is not None else source_key())


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    key = source_key()
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    flags = FLAGS + ["-I", INCLUDE, "-I", CSRC]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc()] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp_path(LIB_PATH) + f".{os.getpid()}.tmp", "w") as f:
        f.write(key + "\n")
    os.replace(stamp_path(LIB_PATH) + f".{os.getpid()}.tmp", stamp_path(LIB_PATH))
    if verbose_ptxas:
        for _, log in results:
            print(log)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    build(force=True, verbose_ptxas="-v" in sys.argv)
    print(LIB_PATH)
