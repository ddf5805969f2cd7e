"""The GEMM kernel's shared-memory plan checked on the CPU (tests/native/tilecfg_check.cpp,
compiled with the host compiler against the library's own header): for every kernel
variant the ring and the epilogue staging fill the data area, the ring keeps at least two
stages, an epilogue chunk is a whole TMA box, and the chunk widths the output tensor maps
use are the ones the kernels stage."""
import ctypes
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA_INC = "/usr/local/cuda/include"


@pytest.fixture(scope="module")
def lib():
    if shutil.which("g++") is None or not os.path.exists(os.path.join(CUDA_INC, "cuda.h")):
        pytest.skip("needs g++ and the CUDA headers")
    out = os.path.join(HERE, "native", "_build")
    os.makedirs(out, exist_ok=True)
    src = os.path.join(HERE, "native", "tilecfg_check.cpp")
    so = os.path.join(out, f"libtilecfg_check.{os.getpid()}.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
                    "-I", os.path.join(ROOT, "mixed_precision_tensor_gb300", "csrc"),
                    "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC, "-o", so, src],
                   check=True)
    L = ctypes.CDLL(so)
    os.remove(so)
    L.tilecfg_violations.restype = ctypes.c_int
    L.chunk_columns.restype = ctypes.c_int
    L.chunk_columns.argtypes = [ctypes.c_int, ctypes.c_int]
    return L


def test_every_variant_fits(lib):
    assert lib.tilecfg_violations() == 0


@pytest.mark.parametrize("out_bytes,c_bufs,cols", [
    (4, 0, 16), (4, 2, 16), (4, 4, 32),      # FP32 out: 8 KiB chunks, 16 KiB with four C buffers
    (2, 0, 32), (2, 2, 32), (2, 4, 64),      # FP16/BF16 out
])
def test_chunk_widths(lib, out_bytes, c_bufs, cols):
    assert lib.chunk_columns(out_bytes, c_bufs) == cols
