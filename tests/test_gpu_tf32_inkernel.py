"""GPU parity of TF32 rounding inside the GEMM kernel (tcg_set_tf32_rounding mode 2).

The GEMM kernel's epilogue warps round op(A) and op(B) to TF32 (nearest even) into the
K-major workspace copies while the kernel multiplies, and the producer waits for each
chunk of K before loading it.  The rounded values, the copies and the accumulation are
those of the pre-pass path, so the result must be the same bit for bit -- and it is
checked the same way: bit-exact against the exact oracle on integer inputs, within the
error bound of "NVIDIA Tensor Core混合精度计算原理与应用解析" section 2.3 on random ones,
bit-exact against the block-FMA model (oracle.MODEL), and bit-identical to the pre-pass
path (mode 1).  Shapes span several K chunks (1024 elements) with ragged ends, every op
combination (K-major sources rounded in place order, M/N-major ones transposed), both
kernel variants, beta != 0 (the epilogue's C loads then stay within a tile), batches
with a shared operand, split-K and tail-split work units.
"""
import numpy as np
import pytest
import torch

import mixed_precision_tensor_gb300 as tcg
import oracle
from helpers import values_equal
from mixed_precision_tensor_gb300 import workloads as wl
from test_gpu_parity import (_assert_results, _check_sampled, _plan, _run_workload,
                             _tie_patterns, run_colmajor)

pytestmark = pytest.mark.gpu

N, T = tcg.TCG_OP_N, tcg.TCG_OP_T
PREPASS, INKERNEL = 1, 2


def _handle(cta_group=2, mode=INKERNEL):
    h = tcg.Handle()
    tcg.check(tcg.tcg_set_kernel_options(h.h, cta_group, 0))
    tcg.check(tcg.tcg_set_tf32_rounding(h.h, mode))
    return h


@pytest.fixture(scope="module", params=[1, 2], ids=["1sm", "2sm"])
def inkernel(cuda_device, request):
    h = _handle(request.param)
    yield h
    h.close()


def test_mode_is_validated(cuda_device):
    h = tcg.Handle()
    for bad in (-1, 3):
        assert tcg.tcg_set_tf32_rounding(h.h, bad) == tcg.TCG_STATUS_INVALID_VALUE
    for ok in (0, 1, 2):
        assert tcg.tcg_set_tf32_rounding(h.h, ok) == tcg.TCG_STATUS_SUCCESS
    h.close()


SHAPES = [(1, 1, 1), (7, 17, 515), (129, 255, 1100), (300, 513, 2049), (257, 260, 4099),
          (64, 8, 640), (520, 130, 1536)]


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("transa,transb", [(N, N), (T, N), (N, T), (T, T)])
def test_inkernel_rounding_integer_and_random(inkernel, m, n, k, transa, transb):
    for dist in ("integer", "uniform"):
        res, guards = run_colmajor(inkernel, transa, transb, m, n, k, 1.0, 0.0, "f32", "f32",
                                   seed=m * 3 + n + k + 7 * transa + 13 * transb, dist=dist)
        assert guards
        _assert_results(res, k, 1.0, 0.0, "f32", exact=(dist == "integer"))


@pytest.mark.parametrize("k", [300, 2500])      # four C buffers (k <= 1024) and two
@pytest.mark.parametrize("transa,transb", [(N, T), (T, N)])
def test_inkernel_rounding_with_beta_batched(inkernel, k, transa, transb):
    for dist in ("integer", "uniform"):
        res, guards = run_colmajor(inkernel, transa, transb, 300, 270, k, 0.5, -1.0, "f32",
                                   "f32", seed=k + transa, dist=dist, batch=3, extra_ld=1)
        assert guards
        _assert_results(res, k, 0.5, -1.0, "f32", exact=(dist == "integer"))


def _colmajor_call(h, transa, transb, m, n, k, A, lda, sA, B, ldb, sB, C, ldc, sC, batch,
                   alpha=1.0, beta=0.0):
    tcg.check(tcg.tcg_gemm_strided_batched(
        h.h, transa, transb, m, n, k, alpha, A, tcg.TCG_R_32F, lda, sA, B, tcg.TCG_R_32F, ldb,
        sB, beta, C, tcg.TCG_R_32F, ldc, sC, batch, tcg.TCG_COMPUTE_32F_FAST_TF32), "gemm")
    tcg.check(tcg.tcg_get_device_error(h.h), "device error")


@pytest.mark.parametrize("transa,transb", [(N, N), (T, N), (N, T), (T, T)])
def test_inkernel_matches_prepass_bit_for_bit(cuda_device, transa, transb):
    """Random FP32 data over more than one wave of tiles and 10 K chunks: the in-kernel
    path's D equals the pre-pass path's (modes 1 and 0) bit for bit: both round with the
    same rule into the same copies."""
    m, n, k = 2560, 2100, 5000                  # 10 x 9 tiles: more than one wave
    rng = np.random.default_rng(5 + transa * 2 + transb)
    dev = torch.device("cuda:0")
    a_rows, a_cols = (m, k) if transa == N else (k, m)
    b_rows, b_cols = (k, n) if transb == N else (n, k)
    A = torch.from_numpy(rng.standard_normal(a_rows * a_cols).astype(np.float32)).to(dev)
    B = torch.from_numpy(rng.standard_normal(b_rows * b_cols).astype(np.float32)).to(dev)
    outs = []
    for mode in (PREPASS, INKERNEL, 0):
        h = _handle(2, mode)
        C = torch.full((m * n,), float("nan"), device=dev)
        _colmajor_call(h, transa, transb, m, n, k, A, a_rows, 0, B, b_rows, 0, C, m, 0, 1)
        outs.append(C.cpu().numpy().view(np.uint32))
        h.close()
    assert np.array_equal(outs[0], outs[1]), "in-kernel rounding differs from the pre-pass"
    assert np.array_equal(outs[0], outs[2])


def test_inkernel_shared_operand_batch(cuda_device):
    """A batch stride of 0 (A shared by all entries): the shared operand is rounded once
    and every entry reads it; integer data, against numpy's int64 product."""
    m, n, k, batch = 200, 264, 1300, 5
    rng = np.random.default_rng(11)
    dev = torch.device("cuda:0")
    A = rng.integers(-2, 3, (k, m)).astype(np.float32)           # column-major m x k: lda = m
    B = rng.integers(-2, 3, (batch, n, k)).astype(np.float32)    # column-major k x n: ldb = k
    h = _handle(2, INKERNEL)
    dA = torch.from_numpy(A.reshape(-1)).to(dev)
    dB = torch.from_numpy(B.reshape(-1)).to(dev)
    C = torch.zeros(batch * m * n, device=dev)
    _colmajor_call(h, N, N, m, n, k, dA, m, 0, dB, k, n * k, C, m, m * n, batch)
    got = C.cpu().numpy().reshape(batch, n, m)                    # D^T per entry
    for b in range(batch):
        want = (A.T.astype(np.int64) @ B[b].T.astype(np.int64))    # (m, n)
        assert np.array_equal(got[b].T, want.astype(np.float32)), b
    h.close()


@pytest.mark.parametrize("transa,transb", [(N, N), (T, T)])
def test_inkernel_rounding_is_nearest_even(cuda_device, transa, transb):
    """Ties, values beside ties and subnormals reach the tensor core rounded to nearest
    even through the in-kernel path too (identity on the other side: D is the rounded
    input), against the oracle's TF32 rounding."""
    rng = np.random.default_rng(91 + 2 * transa + transb)
    m, k = 200, 600
    dev = torch.device("cuda:0")
    h = _handle(2, INKERNEL)
    for side in ("A", "B"):
        vals = _tie_patterns(rng, m * k).reshape(m, k)
        eye = np.eye(k, dtype=np.float32)
        if side == "A":
            M, Nn, Aop, Bop = m, k, vals, eye
        else:
            M, Nn, Aop, Bop = k, m, eye, vals.T.copy()
        Acol = Aop.T.copy() if transa == N else Aop.copy()
        Bcol = Bop.T.copy() if transb == N else Bop.copy()
        lda = M if transa == N else k
        ldb = k if transb == N else Nn
        dA = torch.from_numpy(Acol.reshape(-1)).to(dev)
        dB = torch.from_numpy(Bcol.reshape(-1)).to(dev)
        C = torch.zeros(Nn * M, device=dev)
        _colmajor_call(h, transa, transb, M, Nn, k, dA, lda, 0, dB, ldb, 0, C, M, 0, 1)
        got = C.cpu().numpy().reshape(Nn, M).T
        want = oracle.tf32_round_bits(vals.view(np.uint32)).view(np.float32)
        if side == "B":
            want = want.T
        assert values_equal(got, want), f"operand {side}: not RNE-rounded"
    h.close()


def test_inkernel_split_k(cuda_device):
    """Split-K work units (each a K range of the same tile) walk and wait for only their
    own chunks; within the bound and bit-exact against the model with the same split."""
    h = _handle(2, INKERNEL)
    tcg.check(tcg.tcg_set_split_k(h.h, 5))
    for dist in ("integer", "uniform"):
        res, guards = run_colmajor(h, N, T, 300, 260, 6000, 1.0, 0.0, "f32", "f32",
                                   seed=17, dist=dist)
        assert guards
        _assert_results(res, 6000, 1.0, 0.0, "f32", exact=(dist == "integer"))
    h.close()


@pytest.mark.timeout(900)
def test_inkernel_tail_split(cuda_device):
    """77 tiles on 76 SM pairs, long K: the last tile is cut into K ranges (tail split)
    and the in-kernel path rounds for whole and cut units alike (sampled tiles, corners
    included; the model uses the same per-tile K ranges)."""
    h = _handle(2, INKERNEL)
    w = wl.custom(2816, 1792, 12288, "f32", "f32", 1.0, 0.0, 1, seed=3)
    plan = _plan(h, w)
    assert (plan["plan"][2] > 1).any(), "expected split tail tiles"
    A, B, C = wl.draw(w)
    out = _run_workload(h, w, A, B, C)
    _check_sampled(w, A, B, C, out, exact=False, count=12, model_tiles=6, **plan)
    wi = wl.with_dist(w, "integer")
    A, B, C = wl.draw(wi)
    out = _run_workload(h, wi, A, B, C)
    _check_sampled(wi, A, B, C, out, exact=True, count=6)
    h.close()


def test_inkernel_timeout_is_reported_not_hung(cuda_device):
    """A stage that is never filled (test hook) ends the in-kernel path with TIMEOUT too:
    the epilogue warps stop rounding and leave, and the handle stays usable."""
    h = _handle(2, INKERNEL)
    A = torch.ones(256, 1024, device="cuda")
    B = torch.ones(1024, 256, device="cuda")
    C = torch.zeros(256, 256, device="cuda")
    tcg.check(tcg.tcg_set_debug(h.h, 200_000_000, 1))
    tcg.gemm_rowmajor(h, A, B, C, tf32=True)
    assert tcg.tcg_get_device_error(h.h) == tcg.TCG_STATUS_TIMEOUT
    tcg.check(tcg.tcg_set_debug(h.h, 0, 0))
    tcg.gemm_rowmajor(h, A, B, C, tf32=True)
    assert tcg.tcg_get_device_error(h.h) == tcg.TCG_STATUS_SUCCESS
    torch.cuda.synchronize()
    assert torch.all(C == 1024.0)
    h.close()


def _random_tf32_cases(count=40, seed=20261203):
    """Seeded random TF32 configurations for the in-kernel rounding: shapes up to a few
    hundred with ragged edges and K across up to three 1024-element chunks, op combinations,
    alpha, beta, batches and leading-dimension padding."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(count):
        m, n = (int(x) for x in rng.integers(1, 420, 2))
        k = int(rng.integers(1, 2600))
        transa, transb = (int(x) for x in rng.integers(0, 2, 2))
        alpha = float(rng.choice([1.0, 0.5, -2.0]))
        beta = float(rng.choice([0.0, 1.0, 0.25]))
        batch = int(rng.choice([1, 1, 3]))
        extra_ld = int(rng.integers(0, 2))
        cases.append((i, m, n, k, transa, transb, alpha, beta, batch, extra_ld))
    return cases


@pytest.mark.parametrize("case", _random_tf32_cases(), ids=lambda c: f"cfg{c[0]}")
def test_inkernel_random_configurations(inkernel, case):
    """Within the bound of the exact oracle and bit-exact against the block-FMA model, with
    the guard bands and the ldc padding untouched."""
    i, m, n, k, transa, transb, alpha, beta, batch, extra_ld = case
    res, guards = run_colmajor(inkernel, transa, transb, m, n, k, alpha, beta, "f32", "f32",
                               seed=7000 + i, dist="uniform", extra_ld=extra_ld, batch=batch)
    assert guards, "guard band or ldc padding written"
    _assert_results(res, k, alpha, beta, "f32", exact=False)


# ------------------------------------------------------- the two-word split (3xTF32)
def _split3_call(h, transa, transb, m, n, k, A, B, C, batch=1, alpha=1.0, beta=0.0):
    lda = m if transa == N else k
    ldb = k if transb == N else n
    a_cols = k if transa == N else m
    b_cols = n if transb == N else k
    tcg.check(tcg.tcg_gemm_strided_batched(
        h.h, transa, transb, m, n, k, alpha, A, tcg.TCG_R_32F, lda, lda * a_cols, B,
        tcg.TCG_R_32F, ldb, ldb * b_cols, beta, C, tcg.TCG_R_32F, m, m * n, batch,
        tcg.TCG_COMPUTE_32F_3XTF32), "gemm")
    tcg.check(tcg.tcg_get_device_error(h.h), "device error")


@pytest.mark.parametrize("transa,transb", [(N, N), (T, N), (N, T), (T, T)])
def test_split3_inkernel_matches_prepass_bit_for_bit(cuda_device, transa, transb):
    """The two-word split with both words written by the GEMM kernel: D equals the
    pre-pass path's bit for bit (same high and low words, same three products per K
    slice), over more than one wave of tiles, several K chunks and a batch."""
    m, n, k, batch = 1300, 1800, 3000, 2                      # 6 x 8 tiles per entry
    rng = np.random.default_rng(41 + transa * 2 + transb)
    dev = torch.device("cuda:0")
    A = torch.from_numpy(rng.standard_normal(batch * m * k).astype(np.float32)).to(dev)
    B = torch.from_numpy(rng.standard_normal(batch * k * n).astype(np.float32)).to(dev)
    C0 = torch.from_numpy(rng.standard_normal(batch * m * n).astype(np.float32)).to(dev)
    outs = []
    for mode in (PREPASS, INKERNEL):
        h = _handle(2, mode)
        C = C0.clone()
        _split3_call(h, transa, transb, m, n, k, A, B, C, batch, 0.75, -0.5)
        outs.append(C.cpu().numpy().view(np.uint32))
        h.close()
    assert np.array_equal(outs[0], outs[1]), "in-kernel split differs from the pre-pass"


@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (129, 255, 1100), (300, 520, 2049)])
def test_split3_inkernel_within_fp32_bound(inkernel, m, n, k):
    """Against the oracle's exact product of the FP32 inputs: within
    (k + 8)*2^-23*(|alpha||A||B| + |beta||C|), as for the pre-pass split; integer data
    exact."""
    res, guards = run_colmajor(inkernel, N, T, m, n, k, 0.75, -0.5, "f32", "f32",
                               seed=61 * m + n + k, dist="uniform", split3=True)
    assert guards
    got, D, R, AB, cdec, _ = res[0]
    bound = (k + 8) * 2.0 ** -23 * (0.75 * AB + 0.5 * np.abs(cdec))
    err = np.abs(got.astype(np.float64) - R)
    assert np.all(err <= bound), f"worst {np.max(err / np.maximum(bound, 1e-300))}"
    res, guards = run_colmajor(inkernel, T, N, m, n, k, 1.0, 0.5, "f32", "f32", seed=7 + k,
                               dist="integer", batch=2, split3=True)
    assert guards
    for got, D, R, AB, cdec, _ in res:
        assert values_equal(got.astype(np.float64), R)


def test_split3_default_mode_rounds_in_the_kernel_for_long_k(cuda_device):
    """By default the two-word split with unsplit K >= 6144 rounds inside the GEMM kernel;
    its D equals the pre-pass path's bit for bit (48 tiles, no K split)."""
    m, n, k = 1536, 2048, 8192
    rng = np.random.default_rng(17)
    dev = torch.device("cuda:0")
    A = torch.from_numpy(rng.standard_normal(m * k).astype(np.float32)).to(dev)
    B = torch.from_numpy(rng.standard_normal(k * n).astype(np.float32)).to(dev)
    outs, launches = [], []
    for mode in (PREPASS, 0):
        h = _handle(2, mode)
        C = torch.zeros(m * n, device=dev)
        before = tcg.tcg_launch_count(h.h)
        _split3_call(h, N, N, m, n, k, A, B, C)
        launches.append(tcg.tcg_launch_count(h.h) - before)
        outs.append(C.cpu().numpy().view(np.uint32))
        h.close()
    assert np.array_equal(outs[0], outs[1])
    assert launches[1] < launches[0], launches      # no pre-pass launches by default
