"""The host-buffer entry points (tcg_gemm_ex_host, tcg_gemm_strided_batched_host) against
the device entry points on the same inputs: bit-identical results, untouched ldc padding
and batch gaps in the host C, chunked (pipelined) and single-chunk problems."""
import numpy as np
import pytest
import torch

import mixed_precision_tensor_gb300 as tcg

pytestmark = pytest.mark.gpu

N, T = tcg.TCG_OP_N, tcg.TCG_OP_T
DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
      "e4m3": torch.float8_e4m3fn}
CODE = {"f16": tcg.TCG_R_16F, "bf16": tcg.TCG_R_16BF, "f32": tcg.TCG_R_32F,
        "e4m3": tcg.TCG_R_8F_E4M3}


def _rand(n, t, gen):
    return (torch.rand(n, generator=gen, dtype=torch.float32) * 2 - 1).to(DT[t])


def _bits(x):
    """Raw bits of a tensor for bit-for-bit comparison."""
    x = x.contiguous().cpu()
    return x.view(torch.uint8) if x.element_size() == 1 else (
        x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32))


CASES = [
    # m, n, k, transa, transb, in, out, alpha, beta, extra ld (elements)
    (4096, 4096, 2048, N, N, "f16", "f32", 1.0, 0.0, 0),       # several chunks
    (3000, 2600, 1000, T, T, "bf16", "bf16", 0.5, 1.0, 8),     # 2-D copies of B, ldc padding
    (200, 300, 500, N, T, "f16", "f16", 1.0, 0.5, 8),          # one chunk
    (2048, 4096, 1024, T, N, "f32", "f32", 1.0, -1.0, 0),      # TF32 pre-pass on the device
    (1024, 5120, 512, N, N, "e4m3", "f32", 2.0, 0.0, 16),      # FP8
    (256, 256, 32768, N, N, "f16", "f32", 1.0, 0.0, 0),        # split K, one chunk
    # at least 8 waves of tiles: a grid of D blocks (ragged edges, all op combinations)
    (8192, 5120, 512, N, N, "f16", "f32", 1.0, 0.0, 0),
    (6400, 8192, 256, T, T, "bf16", "bf16", 0.5, 1.0, 8),
    (8192, 6000, 384, N, T, "f16", "f16", 1.0, 0.5, 8),
    (7936, 8192, 256, T, N, "e4m3", "f32", 2.0, 0.0, 16),
]


@pytest.mark.timeout(600)
@pytest.mark.parametrize("m,n,k,ta,tb,in_t,out_t,alpha,beta,xld", CASES)
def test_host_call_matches_device_call(cuda_device, m, n, k, ta, tb, in_t, out_t, alpha, beta,
                                       xld):
    gen = torch.Generator().manual_seed(m + 3 * n + k)
    al = 16 // torch.tensor([], dtype=DT[in_t]).element_size()
    cl = 16 // torch.tensor([], dtype=DT[out_t]).element_size()
    a_rows, a_cols = (m, k) if ta == N else (k, m)
    b_rows, b_cols = (k, n) if tb == N else (n, k)
    lda = -(-a_rows // al) * al + (xld if in_t != "e4m3" else 0)
    ldb = -(-b_rows // al) * al
    ldc = -(-m // cl) * cl + xld
    A = _rand(lda * a_cols, in_t, gen)
    B = _rand(ldb * b_cols, in_t, gen)
    C0 = _rand(ldc * n, out_t, gen)
    comp = tcg.TCG_COMPUTE_32F_FAST_TF32 if in_t == "f32" else tcg.TCG_COMPUTE_32F
    h = tcg.Handle()
    # device call
    dC = C0.clone().cuda()
    tcg.check(tcg.tcg_gemm_ex(h.h, ta, tb, m, n, k, alpha, A.cuda(), CODE[in_t], lda, B.cuda(),
                              CODE[in_t], ldb, beta, dC, CODE[out_t], ldc, comp))
    want = dC.cpu()
    # host call on pinned memory
    hA, hB, hC = A.pin_memory(), B.pin_memory(), C0.clone().pin_memory()
    tcg.check(tcg.tcg_gemm_ex_host(h.h, ta, tb, m, n, k, alpha, hA, CODE[in_t], lda, hB,
                                   CODE[in_t], ldb, beta, hC, CODE[out_t], ldc, comp))
    tcg.check(tcg.tcg_get_device_error(h.h))
    got = hC.clone()
    g = _bits(got).view(n, ldc)
    w = _bits(want).view(n, ldc)
    assert torch.equal(g[:, :m], w[:, :m]), "host call differs from the device call"
    # the ldc padding of the host C holds what it held
    assert torch.equal(g[:, m:], _bits(C0).view(n, ldc)[:, m:])
    # pageable host memory works too
    pC = C0.clone()
    tcg.check(tcg.tcg_gemm_ex_host(h.h, ta, tb, m, n, k, alpha, A, CODE[in_t], lda, B,
                                   CODE[in_t], ldb, beta, pC, CODE[out_t], ldc, comp))
    assert torch.equal(_bits(pC), _bits(got))
    h.close()


BATCHED = [
    # m, n, k, batch, in, out, alpha, beta, gap between batch entries (elements), xld
    (256, 256, 256, 512, "f16", "f16", 1.0, 0.5, 0, 0),          # the batched workload shape
    (130, 200, 96, 40, "bf16", "f32", 1.0, 1.0, 64, 4),          # gaps and ldc padding
    (256, 512, 128, 300, "f16", "f32", 1.0, 0.0, 32, 0),         # gaps, ldc == m
]


@pytest.mark.timeout(600)
@pytest.mark.parametrize("m,n,k,batch,in_t,out_t,alpha,beta,gap,xld", BATCHED)
def test_batched_host_call_matches_device_call(cuda_device, m, n, k, batch, in_t, out_t, alpha,
                                               beta, gap, xld):
    gen = torch.Generator().manual_seed(m + n + k + batch)
    al = 16 // torch.tensor([], dtype=DT[in_t]).element_size()
    cl = 16 // torch.tensor([], dtype=DT[out_t]).element_size()
    lda, ldb = -(-m // al) * al, -(-k // al) * al
    ldc = -(-m // cl) * cl + xld
    sA, sB, sC = lda * k + gap, ldb * n + gap, ldc * n + gap
    A = _rand(sA * batch, in_t, gen)
    B = _rand(sB * batch, in_t, gen)
    C0 = _rand(sC * batch, out_t, gen)
    h = tcg.Handle()
    dC = C0.clone().cuda()
    tcg.check(tcg.tcg_gemm_strided_batched(h.h, N, N, m, n, k, alpha, A.cuda(), CODE[in_t], lda,
                                           sA, B.cuda(), CODE[in_t], ldb, sB, beta, dC,
                                           CODE[out_t], ldc, sC, batch, tcg.TCG_COMPUTE_32F))
    want = dC.cpu()
    hC = C0.clone().pin_memory()
    tcg.check(tcg.tcg_gemm_strided_batched_host(h.h, N, N, m, n, k, alpha, A.pin_memory(),
                                                CODE[in_t], lda, sA, B.pin_memory(),
                                                CODE[in_t], ldb, sB, beta, hC, CODE[out_t], ldc,
                                                sC, batch,
                                                tcg.TCG_COMPUTE_32F))
    tcg.check(tcg.tcg_get_device_error(h.h))
    g, w, c0 = _bits(hC), _bits(want), _bits(C0)
    for b in range(batch):
        blk = slice(b * sC, b * sC + ldc * n)
        gb, wb = g[blk].view(n, ldc), w[blk].view(n, ldc)
        assert torch.equal(gb[:, :m], wb[:, :m]), f"batch entry {b} differs"
        assert torch.equal(gb[:, m:], c0[blk].view(n, ldc)[:, m:])
        if gap:
            gap_blk = slice(b * sC + ldc * n, (b + 1) * sC)
            assert torch.equal(g[gap_blk], c0[gap_blk])
    h.close()


def test_host_call_degenerate_cases(cuda_device):
    h = tcg.Handle()
    C = torch.randn(40, 72).pin_memory()              # column-major 70 x 40, ldc 72
    want = (-1.5 * C[:, :70].double()).float()
    tcg.check(tcg.tcg_gemm_ex_host(h.h, N, N, 70, 40, 0, 1.0, None, tcg.TCG_R_16F, 72, None,
                                   tcg.TCG_R_16F, 64, -1.5, C, tcg.TCG_R_32F, 72,
                                   tcg.TCG_COMPUTE_32F))
    assert torch.equal(C[:, :70], want)
    assert tcg.tcg_gemm_ex_host(h.h, N, N, 0, 40, 8, 1.0, None, tcg.TCG_R_16F, 8, None,
                                tcg.TCG_R_16F, 8, 0.0, C, tcg.TCG_R_32F, 72,
                                tcg.TCG_COMPUTE_32F) == 0
    h.close()


def test_device_call_refuses_host_memory(cuda_device):
    """Device-buffer calls take device memory only: pageable or pinned host memory for an
    operand, the output or the workspace is INVALID_VALUE with nothing launched."""
    h = tcg.Handle()
    F16, F32 = tcg.TCG_R_16F, tcg.TCG_R_32F
    C32, TF32 = tcg.TCG_COMPUTE_32F, tcg.TCG_COMPUTE_32F_FAST_TF32
    SPLIT3 = tcg.TCG_COMPUTE_32F_3XTF32
    INV = tcg.TCG_STATUS_INVALID_VALUE
    dA = torch.ones(64, 64, dtype=torch.float16, device="cuda")
    dB = torch.ones(64, 64, dtype=torch.float16, device="cuda")
    dC = torch.zeros(64, 64, device="cuda")
    for pin in (False, True):
        hX = torch.ones(64, 64, dtype=torch.float16)
        hC = torch.zeros(64, 64)
        if pin:
            hX, hC = hX.pin_memory(), hC.pin_memory()
        before = tcg.tcg_launch_count(h.h)
        for A, B, C in ((hX, dB, dC), (dA, hX, dC), (dA, dB, hC)):
            assert tcg.tcg_gemm_ex(h.h, N, N, 64, 64, 64, 1.0, A, F16, 64, B, F16, 64, 0.0, C,
                                   F32, 64, C32) == INV
        assert tcg.tcg_gemm_ex(h.h, N, N, 64, 64, 0, 1.0, None, F16, 64, None, F16, 64, 2.0, hC,
                               F32, 64, C32) == INV            # D = beta*C alone checks C too
        assert tcg.tcg_gemm_strided_batched(h.h, N, N, 64, 64, 64, 1.0, dA, F16, 64, 0, hX, F16,
                                            64, 0, 0.0, dC, F32, 64, 4096, 1, C32) == INV
        assert tcg.tcg_launch_count(h.h) == before
    # the allocation-free TF32 entry point checks on every call
    fA = torch.ones(64, 64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert tcg.tcg_gemm_tf32_noalloc(s, N, N, 64, 64, 64, 1.0, fA, 64, fA, 64, 0.0,
                                     torch.zeros(64, 64).pin_memory(), 64) == INV
    # a workspace in pinned host memory is refused when a call would use it (the
    # three-product TF32 split writes its rounded operand words there)
    hw = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
    base = (hw.data_ptr() + 255) // 256 * 256
    tcg.check(tcg.tcg_set_workspace(h.h, base, (1 << 20) - 256))
    before = tcg.tcg_launch_count(h.h)
    fC = torch.zeros(64, 64, device="cuda")
    assert tcg.tcg_gemm_ex(h.h, N, N, 64, 64, 64, 1.0, fA, F32, 64, fA, F32, 64, 0.0, fC, F32,
                           64, SPLIT3) == INV
    assert tcg.tcg_launch_count(h.h) == before
    tcg.check(tcg.tcg_set_workspace(h.h, None, 0))
    # device memory still works on the same handle
    tcg.check(tcg.tcg_gemm_ex(h.h, N, N, 64, 64, 64, 1.0, dA, F16, 64, dB, F16, 64, 0.0, dC,
                              F32, 64, C32))
    tcg.check(tcg.tcg_gemm_ex(h.h, N, N, 64, 64, 64, 1.0, fA, F32, 64, fA, F32, 64, 0.0, fC,
                              F32, 64, TF32))
    tcg.check(tcg.tcg_get_device_error(h.h))
    torch.cuda.synchronize()
    assert torch.all(dC == 64.0) and torch.all(fC == 64.0)
    h.close()


def test_clock_probe_reports_the_kernels_sm_clock(cuda_device):
    """The clock probe sums every GEMM CTA's SM cycles and nanoseconds: the ratio is a
    plausible SM clock, it counts only while on, and the results are unchanged."""
    h = tcg.Handle()
    A = torch.ones(1024, 1024, dtype=torch.float16, device="cuda")
    B = torch.ones(1024, 1024, dtype=torch.float16, device="cuda")
    C = torch.zeros(1024, 1024, device="cuda")
    st, cyc, ns = tcg.tcg_read_clock_probe(h.h)
    assert st == tcg.TCG_STATUS_SUCCESS and cyc == 0 and ns == 0       # never enabled
    tcg.check(tcg.tcg_set_clock_probe(h.h, 1))
    for _ in range(3):
        tcg.gemm_rowmajor(h, A, B, C)
    st, cyc, ns = tcg.tcg_read_clock_probe(h.h)
    tcg.check(st)
    assert cyc > 0 and ns > 0
    ghz = cyc / ns
    assert 0.3 < ghz < 2.5, ghz
    tcg.check(tcg.tcg_set_clock_probe(h.h, 0))
    tcg.gemm_rowmajor(h, A, B, C)
    st, cyc2, ns2 = tcg.tcg_read_clock_probe(h.h)
    assert (cyc2, ns2) == (cyc, ns)                                   # off: not counted
    torch.cuda.synchronize()
    assert torch.all(C == 1024.0)
    tcg.check(tcg.tcg_get_device_error(h.h))
    h.close()
