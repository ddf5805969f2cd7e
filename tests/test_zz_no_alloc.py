"""The allocation-free TF32 entry point (tcg_gemm_tf32_noalloc) against the
regular one (tcg_gemm_ex with a workspace) and against the oracle.

Some callers cannot allocate device memory when they multiply (latency-critical
loops, processes whose device memory belongs to another allocator); for them the
library keeps the TF32 path's scratch in a fixed array compiled into it.  This
file checks, through the C ABI, on calls made one after another: the regular
entry point's results within the tests' usual bound; the exact oracle's D within
the same bound; and the block-FMA model bit for bit (the allocation-free call
never splits K, so every tile is one accumulation over all of K).  All four op
combinations run.  It also checks that the calls' error word reads clear and that
problems too large for the fixed array are refused before any device work.  It
sits in its own file, collected last, so that a failure here cannot hide the
other tests' results.
"""
import numpy as np
import pytest
import torch

import mixed_precision_tensor_gb300 as tcg
import oracle
from helpers import check_bound

pytestmark = pytest.mark.gpu

N, T = tcg.TCG_OP_N, tcg.TCG_OP_T
F32, TF32 = tcg.TCG_R_32F, tcg.TCG_COMPUTE_32F_FAST_TF32


def _case(seed, transa, transb, m, n, k, alpha, beta, extra_ld=4):
    rng = np.random.default_rng(seed)
    a_rows, a_cols = (m, k) if transa == N else (k, m)
    b_rows, b_cols = (k, n) if transb == N else (n, k)
    def up4(x):                                       # 16-byte leading dimensions
        return (x + 3) // 4 * 4
    lda, ldb, ldc = up4(a_rows) + extra_ld, up4(b_rows) + extra_ld, up4(m) + extra_ld
    A = rng.uniform(-1, 1, lda * a_cols).astype(np.float32)
    B = rng.uniform(-1, 1, ldb * b_cols).astype(np.float32)
    C = rng.standard_normal(ldc * n).astype(np.float32)
    return dict(transa=transa, transb=transb, m=m, n=n, k=k, alpha=alpha, beta=beta, A=A, B=B,
                C=C, lda=lda, ldb=ldb, ldc=ldc)


def _run_regular(h, c):
    dev = torch.device("cuda:0")
    dA, dB = torch.from_numpy(c["A"]).to(dev), torch.from_numpy(c["B"]).to(dev)
    dC = torch.from_numpy(c["C"]).to(dev)
    tcg.check(tcg.tcg_gemm_ex(h.h, c["transa"], c["transb"], c["m"], c["n"], c["k"], c["alpha"],
                              dA, F32, c["lda"], dB, F32, c["ldb"], c["beta"], dC, F32, c["ldc"],
                              TF32))
    tcg.check(tcg.tcg_get_device_error(h.h))
    return dC.cpu().numpy()


def _run_noalloc(c, stream):
    dev = torch.device("cuda:0")
    dA, dB = torch.from_numpy(c["A"]).to(dev), torch.from_numpy(c["B"]).to(dev)
    dC = torch.from_numpy(c["C"]).to(dev)
    torch.cuda.synchronize()
    s = tcg.tcg_gemm_tf32_noalloc(stream.cuda_stream, c["transa"], c["transb"], c["m"], c["n"],
                                  c["k"], c["alpha"], dA, c["lda"], dB, c["ldb"], c["beta"], dC,
                                  c["ldc"])
    tcg.check(s, "tcg_gemm_tf32_noalloc")
    stream.synchronize()
    return dC.cpu().numpy()


def _block(x, c):
    return x[: c["ldc"] * c["n"]].reshape(c["n"], c["ldc"])[:, : c["m"]].T.astype(np.float64)


def test_noalloc_matches_regular_entry_point_and_oracle(cuda_device):
    h = tcg.Handle()
    stream = torch.cuda.Stream()
    cases = [_case(101, N, N, 300, 520, 333, 0.75, -0.5),
             _case(202, T, N, 1024, 768, 2048, 1.0, 1.0),
             _case(303, N, T, 257, 129, 100, 1.0, 0.0),
             _case(404, T, T, 640, 384, 520, -2.0, 0.25)]
    for c in cases:                                   # calls one after another
        want = _run_regular(h, c)
        got = _run_noalloc(c, stream)
        args = (c["transa"], c["transb"], c["m"], c["n"], c["k"], c["alpha"], c["A"], oracle.F32,
                c["lda"], c["B"], oracle.F32, c["ldb"], c["beta"], c["C"], oracle.F32, c["ldc"])
        D, _, absab = oracle.gemm(*args, tf32=True, want_r=False)
        cval = _block(c["C"], c)
        # the regular entry point's result, within the parity tests' bound
        ok, worst, _ = check_bound(_block(got, c), _block(want, c), absab, cval,
                                   c["k"], c["alpha"], c["beta"], "f32")
        assert ok, f"against tcg_gemm_ex: worst normalised difference {worst}"
        # the exact oracle's D, within the same bound
        ok, worst, _ = check_bound(_block(got, c), D.astype(np.float64), absab, cval,
                                   c["k"], c["alpha"], c["beta"], "f32")
        assert ok, f"against the oracle: worst normalised error {worst}"
        # the block-FMA model, bit for bit: one accumulation over all of K per tile
        Dm = oracle.gemm_model(*args, tf32=True, **oracle.MODEL[oracle.F32])
        g = _block(got, c)
        same = (g == Dm) | (np.isnan(g) & np.isnan(Dm))
        assert same.all(), f"{int((~same).sum())} elements differ from the block-FMA model"
        # the ldc padding rows are never written
        pad_in = c["C"][: c["ldc"] * c["n"]].reshape(c["n"], c["ldc"])[:, c["m"]:]
        pad_out = got[: c["ldc"] * c["n"]].reshape(c["n"], c["ldc"])[:, c["m"]:]
        assert np.array_equal(pad_in, pad_out)
    assert tcg.tcg_noalloc_device_error(stream.cuda_stream) == tcg.TCG_STATUS_SUCCESS
    h.close()


def test_noalloc_refuses_problems_beyond_its_scratch(cuda_device):
    m = n = 2048
    k = 2056                   # (2048 + 2048) * 2056 * 4 bytes > 32 MiB
    dA = torch.zeros(m * k, device="cuda")
    dB = torch.zeros(k * n, device="cuda")
    dC = torch.full((m * n,), 3.0, device="cuda")
    s = tcg.tcg_gemm_tf32_noalloc(None, N, N, m, n, k, 1.0, dA, m, dB, k, 0.0, dC, m)
    assert s == tcg.TCG_STATUS_NOT_SUPPORTED
    torch.cuda.synchronize()
    assert torch.all(dC == 3.0)                        # nothing ran
