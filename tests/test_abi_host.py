"""C-ABI tests that need no GPU: the library loads, exports every symbol that
include/tcg.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import mixed_precision_tensor_gb300 as tcg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mixed_precision_tensor_gb300 import _build
    _build.build()
    return tcg.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "tcg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tcg_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_symbols()
    for required in ("tcg_create", "tcg_destroy", "tcg_set_stream", "tcg_gemm_ex",
                     "tcg_gemm_strided_batched", "tcg_get_device_error", "tcg_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) <= set(tcg.EXPORTS)


def test_status_strings(lib):
    assert tcg.tcg_status_string(0) == "TCG_STATUS_SUCCESS"
    assert tcg.tcg_status_string(6) == "TCG_STATUS_TIMEOUT"
    assert tcg.tcg_status_string(99) == "TCG_STATUS_UNKNOWN"


@pytest.fixture
def handle(lib):
    h = tcg.tcg_create()
    yield h
    assert tcg.tcg_destroy(h) == tcg.TCG_STATUS_SUCCESS


# Fake, 16-byte aligned "device" addresses: the checks must reject the call before
# anything dereferences them.
PA, PB, PC = 0x10000, 0x20000, 0x30000
F16, BF16, F32 = tcg.TCG_R_16F, tcg.TCG_R_16BF, tcg.TCG_R_32F
E4M3, E5M2 = tcg.TCG_R_8F_E4M3, tcg.TCG_R_8F_E5M2
N, T = tcg.TCG_OP_N, tcg.TCG_OP_T
C32, TF32, SPLIT3 = (tcg.TCG_COMPUTE_32F, tcg.TCG_COMPUTE_32F_FAST_TF32,
                     tcg.TCG_COMPUTE_32F_3XTF32)
INV, NSUP = tcg.TCG_STATUS_INVALID_VALUE, tcg.TCG_STATUS_NOT_SUPPORTED


def gemm(h, transa=N, transb=N, m=64, n=64, k=64, alpha=1.0, A=PA, at=F16, lda=64, B=PB,
         bt=F16, ldb=64, beta=0.0, C=PC, ct=F32, ldc=64, comp=C32):
    return tcg.tcg_gemm_ex(h, transa, transb, m, n, k, alpha, A, at, lda, B, bt, ldb, beta, C,
                           ct, ldc, comp)


@pytest.mark.parametrize("kw,status", [
    (dict(m=-1), INV), (dict(n=-1), INV), (dict(k=-1), INV),
    (dict(transa=2), INV), (dict(transb=-1), INV),
    (dict(at=7), INV), (dict(ct=9), INV), (dict(comp=5), INV),
    (dict(lda=63), INV),                      # lda < m for OP_N
    (dict(transa=T, m=128, k=64, lda=56, ldc=128), INV),  # OP_T: lda < k
    (dict(transb=T, n=128, ldb=64), INV),                 # OP_T: ldb < n
    (dict(ldb=60), INV),                      # ldb < k
    (dict(ldc=32), INV),                      # ldc < m
    (dict(m=60, lda=68, ldc=68), INV),        # 68*2 bytes = 136, not a multiple of 16
    (dict(ldc=66), INV),                      # 66*4 bytes: multiple of 8 only
    (dict(A=PA + 8), INV),                    # misaligned pointer
    (dict(B=PB + 2), INV),
    (dict(C=PC + 4), INV),
    (dict(A=None), INV), (dict(B=None), INV), (dict(C=None), INV),
    (dict(at=F16, bt=BF16), NSUP),            # mixed input types
    (dict(at=F32, bt=F32, comp=C32), NSUP),   # FP32 inputs need the TF32 compute type
    (dict(at=F32, bt=F32, comp=TF32, ct=F16, ldc=64), NSUP),
    (dict(at=F16, bt=F16, comp=TF32), NSUP),
    (dict(at=F16, bt=F16, ct=BF16), NSUP),    # 16-bit output must match the input type
    (dict(at=F16, bt=F16, comp=SPLIT3), NSUP),                       # split needs FP32 inputs
    (dict(at=E4M3, bt=E5M2), NSUP),                                  # FP8 A and B alike
    (dict(at=E4M3, bt=E4M3, ct=E4M3, ldc=64), NSUP),                 # FP8 is input-only
    (dict(at=E4M3, bt=E4M3, comp=TF32), NSUP),
    (dict(at=E5M2, bt=E5M2, lda=72), INV),                           # 72 bytes: not 16-byte
    (dict(at=F32, bt=F32, comp=SPLIT3, ct=F16, ldc=64), NSUP),      # and FP32 output
])
def test_argument_checks(handle, kw, status):
    assert gemm(handle, **kw) == status


def test_null_handle_is_invalid(lib):
    assert tcg.tcg_gemm_ex(None, N, N, 1, 1, 1, 1.0, PA, F16, 8, PB, F16, 8, 0.0, PC, F32, 4,
                           C32) == INV
    assert tcg.tcg_get_device_error(None) == INV
    assert tcg.tcg_set_stream(None, None) == INV
    assert tcg.tcg_destroy(None) == INV
    assert lib.tcg_create(None) == INV


def test_empty_problems_are_noops_without_cuda(handle):
    # m == 0 / n == 0 / batch == 0 succeed before any device work (no GPU here)
    assert gemm(handle, m=0, lda=8, ldc=4) == tcg.TCG_STATUS_SUCCESS
    assert gemm(handle, n=0) == tcg.TCG_STATUS_SUCCESS
    s = tcg.tcg_gemm_strided_batched(handle, N, N, 64, 64, 64, 1.0, PA, F16, 64, 4096, PB, F16,
                                     64, 4096, 0.0, PC, F32, 64, 4096, 0, C32)
    assert s == tcg.TCG_STATUS_SUCCESS
    # k == 0 / alpha == 0: A and B are not read, so NULL is fine there
    assert gemm(handle, m=0, k=0, A=None, B=None, lda=8, ldc=4) == tcg.TCG_STATUS_SUCCESS


def test_batched_stride_checks(handle):
    def b(**kw):
        args = dict(sA=4096, sB=4096, sC=4096, batch=4)
        args.update(kw)
        return tcg.tcg_gemm_strided_batched(handle, N, N, 64, 64, 64, 1.0, PA, F16, 64,
                                            args["sA"], PB, F16, 64, args["sB"], 0.0, PC, F32,
                                            64, args["sC"], args["batch"], C32)
    assert b(sA=-8) == INV
    assert b(sA=4100) == INV                   # 4100*2 bytes not a multiple of 16
    assert b(sC=4098) == INV                   # 4098*4 bytes not a multiple of 16
    assert b(sC=0) == INV                      # outputs would alias
    assert b(batch=-1) == INV


def test_workspace_size_query(lib):
    assert tcg.tcg_gemm_workspace_size(N, N, 64, 64, 64, F16, C32) == 0
    ws = tcg.tcg_gemm_workspace_size(N, N, 100, 50, 30, F32, TF32)
    kp = 32
    copies = (100 + 50) * kp * 4             # the rounded K-major copies (256-byte multiples)
    # plus the counters of the in-kernel rounding: (2 items + 1 panel) x 4 bytes per
    # operand, in one 256-byte block
    assert ws == copies + 256
    assert tcg.tcg_gemm_workspace_size(N, N, 100, 50, 30, F32, SPLIT3) == 2 * copies + 256
    assert tcg.tcg_set_workspace(tcg.tcg_create(), 0x1000 + 16, 1024) == INV   # not 256-aligned


def test_debug_hook_and_launch_count(handle):
    assert tcg.tcg_set_debug(handle, 1000, 1) == tcg.TCG_STATUS_SUCCESS
    assert tcg.tcg_set_debug(handle, 0, 0) == tcg.TCG_STATUS_SUCCESS
    assert tcg.tcg_launch_count(handle) == 0
    # a handle that never launched reports no device error, with no CUDA call
    assert tcg.tcg_get_device_error(handle) == tcg.TCG_STATUS_SUCCESS


def test_product_path_has_no_oracle_dependency():
    """The package and the CUDA sources never import or link the oracle."""
    pkg = os.path.join(ROOT, "mixed_precision_tensor_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "tcg_oracle" not in text and "liboracle" not in text, f


def test_split_k_plan_rule():
    # Split only when the tiles fill less than half of the clusters; at least 8 K blocks
    # per range; at most 64 ranges; no empty range.
    plan = lambda *a: tcg.tcg_split_k_plan(*a)
    assert plan(1, 512, 76) == (0, 64, 8)
    assert plan(40, 512, 76)[1:] == (1, 512)            # 80 > 76: the GPU is busy enough
    assert plan(10, 512, 76)[1] == 7                     # 76 // 10
    assert plan(10, 24, 76)[1] == 3                      # at most 24 // 8 ranges
    assert plan(10, 12, 76)[1:] == (1, 12)               # 12 // 8: one range, no split
    assert plan(1, 15, 76)[1:] == (1, 15)                # too short to split
    assert plan(500, 64, 76, 3)[1:] == (3, 22)           # forced
    assert plan(1, 2, 76, 8)[1:] == (2, 1)               # forced, capped by the K blocks
    for tiles in (1, 2, 5, 19, 37):
        for nkb in (1, 4, 9, 33, 100, 1000):
            for forced in (0, 2, 7, 64):
                st, s, kb = plan(tiles, nkb, 76, forced)
                assert st == 0 and 1 <= s <= 64
                assert (s - 1) * kb < nkb <= s * kb          # every range non-empty
                if s == 1:
                    assert kb == nkb


def test_split_k_argument_checks():
    INV = tcg.TCG_STATUS_INVALID_VALUE
    assert tcg.tcg_split_k_plan(-1, 4, 76)[0] == INV
    assert tcg.tcg_split_k_plan(1, 4, 76, 65)[0] == INV
    assert tcg.load_library().tcg_split_k_plan(1, 4, 76, 0, None, None) == INV
    assert tcg.tcg_set_split_k(None, 2) == INV
    assert tcg.tcg_set_tile_n(None, 128) == INV
    h = tcg.tcg_create()
    assert tcg.tcg_set_tile_n(h, 64) == INV and tcg.tcg_set_tile_n(h, 129) == INV
    assert tcg.tcg_set_tile_n(h, 128) == 0 and tcg.tcg_set_tile_n(h, 0) == 0
    tcg.tcg_destroy(h)
    assert tcg.tcg_gemm_split_k(None, 1, 1, 1, tcg.TCG_R_16F, tcg.TCG_COMPUTE_32F)[0] == INV



def test_host_buffer_calls_check_arguments_without_a_gpu():
    INV = tcg.TCG_STATUS_INVALID_VALUE
    lib = tcg.load_library()
    args = (N, N, 16, 16, 16, 1.0, None, tcg.TCG_R_16F, 16, None, tcg.TCG_R_16F, 16, 0.0, None,
            tcg.TCG_R_32F, 16, tcg.TCG_COMPUTE_32F)
    assert lib.tcg_gemm_ex_host(None, *args) == INV
    bargs = (N, N, 16, 16, 16, 1.0, None, tcg.TCG_R_16F, 16, 256, None, tcg.TCG_R_16F, 16, 256,
             0.0, None, tcg.TCG_R_32F, 16, 256, 2, tcg.TCG_COMPUTE_32F)
    assert lib.tcg_gemm_strided_batched_host(None, *bargs) == INV


def test_tail_split_plan_rule():
    # 256 tiles of 146 us (the TF32 4096 x 4096 x 16384 shape) on 76 tile slots: three full
    # waves, the 28 tiles of the partial wave in two K halves (3.5 tile times instead of
    # 4); splitting the last 104 tiles saves as much but reduces four times the partials
    st, full, s, kb = tcg.tcg_tail_split_plan(256, 256, 76, 256 * 1024 / 1.8e3, 262144.0)
    assert (st, full, s, kb) == (0, 228, 2, 128)
    # three times the tensor work per tile (the two-word split): the same plan
    assert tcg.tcg_tail_split_plan(256, 256, 76, 3 * 256 * 1024 / 1.8e3, 262144.0)[1:3] == (228, 2)
    # 1024 tiles of 36 us (8192^3 FP16): the half tile saved does not pay for the partial sums
    assert tcg.tcg_tail_split_plan(1024, 64, 76, 64 * 1024 / 1.8e3, 262144.0)[1:] == (1024, 1, 64)
    # whole waves, or fewer tiles than slots: nothing to split
    assert tcg.tcg_tail_split_plan(152, 256, 76, 145.6, 262144.0)[2] == 1
    assert tcg.tcg_tail_split_plan(50, 256, 76, 145.6, 262144.0)[2] == 1
    # too few K blocks to cut
    assert tcg.tcg_tail_split_plan(100, 3, 76, 1.0e4, 262144.0)[2] == 1
    # every range non-empty
    for tiles in (77, 100, 153, 400):
        for nkb in (4, 9, 64, 300):
            st, full, s, kb = tcg.tcg_tail_split_plan(tiles, nkb, 76, 1.0e5, 262144.0)
            assert st == 0 and 0 <= full <= tiles and full % 76 == 0
            assert (s - 1) * kb < nkb <= s * kb
    assert tcg.tcg_tail_split_plan(-1, 4, 76, 1.0, 1.0)[0] == tcg.TCG_STATUS_INVALID_VALUE



def test_gemm_rowmajor_argument_checks(lib):
    """The row-major convenience refuses operands that the pointer-level call would
    misread (shapes, dtypes, layout, placement) before calling the library."""
    import torch
    h = tcg.Handle()
    f16 = torch.float16
    A, B, C = torch.zeros(8, 16, dtype=f16), torch.zeros(16, 24, dtype=f16), torch.zeros(8, 24)
    bad = [
        (A, torch.zeros(12, 24, dtype=f16), C, {}),                       # inner sizes differ
        (A, B, torch.zeros(8, 16), {}),                                   # wrong output shape
        (A, B.to(torch.bfloat16), C, {}),                                 # A, B dtypes differ
        (A, torch.zeros(24, 16, dtype=f16).t(), C, {}),                   # not contiguous
        (A[None], B, C[None], {}),                                        # 3-D with 2-D
        (A[None].expand(2, 8, 16), B[None].expand(2, 16, 24), C[None].expand(2, 8, 24), {}),
        (A[None], B[None].repeat(2, 1, 1), C[None], {}),                  # batch sizes differ
        (A, B, C, {}),                                                    # CPU tensors, device call
    ]
    for a, b, c, kw in bad:
        with pytest.raises(ValueError):
            tcg.gemm_rowmajor(h, a, b, c, **kw)
    h.close()


def test_size_limits_are_not_supported(handle):
    """The kernels index tiles and TMA coordinates with 32-bit integers: sizes past
    2^31 - 1, or more than 2^31 - 1 tiles in one call, are refused (NOT_SUPPORTED) by the
    host checks, before any CUDA call."""
    big = 1 << 31
    assert gemm(handle, m=big, lda=big, ldc=big) == NSUP
    assert gemm(handle, n=big) == NSUP
    assert gemm(handle, k=big, ldb=big) == NSUP
    # 2 x 1 tiles per entry (128-row tiles) times 2^31 - 1 entries
    lim = big - 1
    assert tcg.tcg_gemm_strided_batched(handle, N, N, 256, 256, 64, 1.0, PA, F16, 256, 0, PB,
                                        F16, 64, 0, 0.0, PC, F32, 256, 65536, lim, C32) == NSUP
    # inside the limits the size checks pass it on: with no device the call then fails to
    # bind one, and on a GPU machine the pointer check refuses these stand-in addresses
    st = tcg.tcg_gemm_strided_batched(handle, N, N, 256, 256, 64, 1.0, PA, F16, 256, 0, PB,
                                      F16, 64, 0, 0.0, PC, F32, 256, 65536, 1 << 20, C32)
    assert st != NSUP
