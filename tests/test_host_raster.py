"""The GEMM kernel's tile rasterisation (tcg::raster, a host-and-device function in
csrc/tcg_internal.h) checked on the CPU: every tile of every batch entry is visited
exactly once, batch entries in order, and consecutive tiles walk a group of group_m
m-tiles column by column (tests/native/raster_check.cpp, compiled with the host
compiler against the library's own header)."""
import ctypes
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA_INC = "/usr/local/cuda/include"


def _build():
    if shutil.which("g++") is None or not os.path.exists(os.path.join(CUDA_INC, "cuda.h")):
        pytest.skip("needs g++ and the CUDA headers")
    out = os.path.join(HERE, "native", "_build")
    os.makedirs(out, exist_ok=True)
    src = os.path.join(HERE, "native", "raster_check.cpp")
    hdr = os.path.join(ROOT, "mixed_precision_tensor_gb300", "csrc", "tcg_internal.h")
    lib = os.path.join(out, "libraster_check.so")
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(src),
                                                              os.path.getmtime(hdr)):
        tmp = lib + f".{os.getpid()}.tmp"
        subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                        "-I", os.path.join(ROOT, "mixed_precision_tensor_gb300", "csrc"),
                        "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC, "-o", tmp, src],
                       check=True)
        os.replace(tmp, lib)
    f = ctypes.CDLL(lib).raster_mismatches
    f.restype = ctypes.c_int64
    f.argtypes = [ctypes.c_int] * 4
    return f


@pytest.mark.parametrize("m_tiles,n_tiles,batch,group_m", [
    (32, 32, 1, 8),       # 8192^3 on SM pairs (256 x 256 tiles)
    (64, 16, 1, 8),       # 16384 x 4096 output
    (16, 16, 1, 8),       # 4096 x 4096 output
    (1, 1, 512, 8),       # 512 batch entries of one tile
    (1, 2, 512, 8),       # the same with narrow (256 x 128) tiles
    (33, 17, 2, 4),       # ragged group at the bottom, two batch entries
    (7, 5, 3, 8),         # fewer m-tiles than a group
    (5, 9, 1, 1),         # group of one: plain column order
    (40, 3, 1, 16),
])
def test_raster_is_a_grouped_bijection(m_tiles, n_tiles, batch, group_m):
    assert _build()(m_tiles, n_tiles, batch, group_m) == 0
