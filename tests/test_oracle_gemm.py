"""Pins of the oracle GEMM (CPU only).

The oracle is held to things other than itself: closed forms (all-ones and
identity operands), exact integer arithmetic (numpy int64 matmul), exact
rational arithmetic (fractions.Fraction) on 16x16x16, the worked vectors of
"NVIDIA Tensor Core混合精度计算原理与应用解析" sections 2.2.1 and 2.2.3
(tests/golden/), and numpy float64 matmul.  A dropped alpha/beta term, a wrong
sign, a transposed operand or a wrong leading dimension fails at least one of
them (the op-flag cases use non-square shapes and padded leading dimensions).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from helpers import TYPE_CODE, load_golden, oracle_rowmajor, raw
from mixed_precision_tensor_gb300 import workloads as wl


def _store(x64, t):
    """FP64 values that are exact in type t -> raw storage array."""
    if t in ("e4m3", "e5m2"):
        import torch
        dt = torch.float8_e4m3fn if t == "e4m3" else torch.float8_e5m2
        return torch.from_numpy(np.asarray(x64, dtype=np.float32)).to(dt).view(torch.uint8).numpy()
    if t == "f16":
        return x64.astype(np.float16).view(np.uint16)
    if t == "bf16":
        return oracle.f64_to_bf16_bits(x64)
    return x64.astype(np.float32)


def _colmajor(x2d):
    """Flat column-major storage of a 2-D array (element (i, j) at i + j*rows)."""
    return np.asfortranarray(x2d).reshape(-1, order="F")


@pytest.mark.parametrize("t", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("k", [1, 3, 16, 255, 1024, 2048, 4096])
def test_all_ones_gives_k(t, k):
    m, n = 5, 7
    A = _store(np.ones(m * k), t)
    B = _store(np.ones(k * n), t)
    D, R, AB = oracle.gemm(oracle.OP_N, oracle.OP_N, m, n, k, 1.0, A, TYPE_CODE[t], m, B,
                           TYPE_CODE[t], k, 0.0, None, oracle.F32, m, tf32=(t == "f32"))
    assert np.all(D == np.float32(k))
    assert np.all(AB == k)
    if k <= 2048:
        D16, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, m, n, k, 1.0, A, TYPE_CODE[t], m, B,
                                TYPE_CODE[t], k, 0.0, None, oracle.F16, m, tf32=(t == "f32"))
        assert np.all(D16.view(np.float16) == np.float16(k))


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
def test_identity_gives_rounded_alpha_b_plus_beta_c(out):
    rng = np.random.default_rng(11)
    k, n = 40, 24
    alpha, beta = 0.375, -1.5
    I = _store(np.eye(k).reshape(-1, order="F"), "f16")
    Bv = rng.uniform(-4, 4, (k, n)).astype(np.float16).astype(np.float64)
    Cv = rng.standard_normal((k, n))
    if out == "f16":
        C = Cv.astype(np.float16)
        Cd = C.astype(np.float64)
        Craw = _colmajor(C).view(np.uint16)
    elif out == "bf16":
        Craw = oracle.f64_to_bf16_bits(_colmajor(Cv))
        Cd = oracle.bf16_to_f64(Craw).reshape(k, n, order="F")
    else:
        C = Cv.astype(np.float32)
        Cd = C.astype(np.float64)
        Craw = _colmajor(C)
    D, R, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, k, n, k, alpha, I, oracle.F16, k,
                          _store(_colmajor(Bv), "f16"), oracle.F16, k, beta, Craw,
                          TYPE_CODE[out], k)
    exact = alpha * Bv + beta * Cd                   # exact in FP64
    assert np.array_equal(R, exact)
    if out == "f32":
        assert np.array_equal(D.view(np.uint32), exact.astype(np.float32).view(np.uint32))
    elif out == "f16":
        assert np.array_equal(D.view(np.uint16), exact.astype(np.float16).view(np.uint16))
    else:
        import torch
        want = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16)
        # exact values here have <= 24 significant bits, so float32 is exact
        assert np.array_equal(D.view(np.uint16),
                              want.view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("transa", [oracle.OP_N, oracle.OP_T])
@pytest.mark.parametrize("transb", [oracle.OP_N, oracle.OP_T])
@pytest.mark.parametrize("t", ["f16", "bf16", "f32", "e4m3", "e5m2"])
def test_small_integers_exact_against_int64_matmul(transa, transb, t):
    rng = np.random.default_rng(12 + 2 * transa + transb)
    m, n, k = 37, 29, 53
    pad = 3
    opA = rng.integers(-2, 3, (m, k))
    opB = rng.integers(-2, 3, (k, n))
    Cint = rng.integers(-8, 9, (m, n))
    alpha, beta = 2.0, -3.0
    # store op(A) as A (N: m x k, ld >= m) or A^T (T: k x m, ld >= k), with padding rows
    def stored(op, trans, rows, cols):
        mat = op if trans == oracle.OP_N else op.T
        ld = mat.shape[0] + pad
        buf = np.full((ld, mat.shape[1]), 99, dtype=np.int64)   # junk in the padding
        buf[: mat.shape[0]] = mat
        return _colmajor(buf), ld
    Af, lda = stored(opA, transa, m, k)
    Bf, ldb = stored(opB, transb, k, n)
    ldc = m + pad
    Cbuf = np.full((ldc, n), 1e30)
    Cbuf[:m] = Cint
    D, R, AB = oracle.gemm(transa, transb, m, n, k, alpha, _store(Af.astype(np.float64), t),
                           TYPE_CODE[t], lda, _store(Bf.astype(np.float64), t), TYPE_CODE[t],
                           ldb, beta, _colmajor(Cbuf).astype(np.float32), oracle.F32, ldc,
                           tf32=(t == "f32"))
    want = 2 * (opA @ opB) - 3 * Cint
    assert np.array_equal(R, want.astype(np.float64))
    assert np.array_equal(D, want.astype(np.float32))
    assert np.array_equal(AB, (np.abs(opA) @ np.abs(opB)).astype(np.float64))


def test_rowmajor_mapping_matches_numpy_matmul():
    w = wl.custom(33, 21, 45, "f16", "f32", alpha=1.0, beta=1.0, seed=5, dist="integer")
    A, B, C = wl.draw(w)
    D, R, _ = oracle_rowmajor(w, A, B, C)
    want = A[0].astype(np.int64) @ B[0].astype(np.int64) + C[0].astype(np.float64)
    assert np.array_equal(R, want)
    # a sub-block equals the same block of the full result
    Db, _, _ = oracle_rowmajor(w, A, B, C, rows=(7, 30), cols=(3, 11))
    assert np.array_equal(Db, D[7:30, 3:11])


def _rne_from_fraction_via_double(x: Fraction, kind: str):
    """One correctly rounded conversion of an exact rational: float(Fraction) is
    correctly rounded to FP64; the result is returned with a flag telling whether
    the exact value lies within 2^-48 (relative) of a rounding midpoint of the
    target type, where the FP64 step could double-round."""
    d = float(x)
    if kind == "f32":
        r = np.float32(d)
        lo = np.nextafter(r, np.float32(-np.inf), dtype=np.float32)
        hi = np.nextafter(r, np.float32(np.inf), dtype=np.float32)
    else:
        r = np.float16(d)
        lo = np.nextafter(r, np.float16(-np.inf), dtype=np.float16)
        hi = np.nextafter(r, np.float16(np.inf), dtype=np.float16)
    mids = [(Fraction(float(r)) + Fraction(float(lo))) / 2, (Fraction(float(r)) + Fraction(float(hi))) / 2]
    tol = abs(x) * Fraction(1, 2 ** 48)
    # the FP64 step is exact when x fits in FP64: then no double rounding is possible
    risky = Fraction(d) != x and any(abs(x - mid) <= tol for mid in mids)
    return r, risky


@pytest.mark.parametrize("t,out", [("f16", "f32"), ("f16", "f16"), ("bf16", "f32"),
                                   ("f32", "f32")])
def test_bruteforce_16x16x16_exact_rational(t, out):
    rng = np.random.default_rng(13)
    m = n = k = 16
    alpha, beta = 0.75, -1.25
    Av = rng.uniform(-1, 1, (m, k))
    Bv = rng.uniform(-1, 1, (k, n))
    Cv = rng.standard_normal((m, n))
    if t == "f32":
        Araw = _colmajor(Av).astype(np.float32)
        Braw = _colmajor(Bv).astype(np.float32)
        # TF32 inputs: round with the integer-bit formulation pinned in
        # test_oracle_formats (independent of the oracle's FP64 routine)
        def t32(a):
            u = a.view(np.uint32).astype(np.uint64)
            return (((u + 0xFFF + ((u >> 13) & 1)) & 0xFFFFE000).astype(np.uint32)).view(np.float32)
        Aq = t32(Araw).astype(np.float64).reshape(m, k, order="F")
        Bq = t32(Braw).astype(np.float64).reshape(k, n, order="F")
    else:
        Araw = _store(_colmajor(Av).astype(np.float32).astype(np.float64) if t == "bf16" else
                      _colmajor(Av).astype(np.float16).astype(np.float64), t)
        Braw = _store(_colmajor(Bv).astype(np.float32).astype(np.float64) if t == "bf16" else
                      _colmajor(Bv).astype(np.float16).astype(np.float64), t)
        dec = oracle.f16_to_f64 if t == "f16" else oracle.bf16_to_f64
        Aq = dec(Araw).reshape(m, k, order="F") if t == "bf16" else \
            Araw.view(np.float16).astype(np.float64).reshape(m, k, order="F")
        Bq = dec(Braw).reshape(k, n, order="F") if t == "bf16" else \
            Braw.view(np.float16).astype(np.float64).reshape(k, n, order="F")
    if out == "f16":
        Craw = _colmajor(Cv).astype(np.float16)
        Cq = Craw.astype(np.float64).reshape(m, n, order="F")
        Craw = Craw.view(np.uint16)
    else:
        Craw = _colmajor(Cv).astype(np.float32)
        Cq = Craw.astype(np.float64).reshape(m, n, order="F")
    D, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, m, n, k, alpha, Araw, TYPE_CODE[t], m, Braw,
                          TYPE_CODE[t], k, beta, Craw, TYPE_CODE[out], m, tf32=(t == "f32"))
    Dv = D.view(np.float16) if out == "f16" else D
    checked = 0
    for i in range(m):
        for j in range(n):
            s = sum(Fraction(Aq[i, p]) * Fraction(Bq[p, j]) for p in range(k))
            x = Fraction(alpha) * s + Fraction(beta) * Fraction(Cq[i, j])
            want, risky = _rne_from_fraction_via_double(x, out)
            if risky:
                continue
            checked += 1
            assert Dv[i, j] == want, (i, j, float(x), Dv[i, j], want)
    assert checked >= 250


def _golden_case(name, t):
    g = load_golden(name)
    k = int(g["k"])
    a = np.array([float(v) for v in g["a"]])
    b = np.array([float(v) for v in g["b"]])
    A = _store(a, t)           # 1 x k, lda = 1
    B = _store(b, t)           # k x 1, ldb = k
    # exact in the input type (checked)
    if t == "f16":
        assert np.array_equal(A.view(np.float16).astype(np.float64), a)
    elif t == "bf16":
        assert np.array_equal(oracle.bf16_to_f64(A), a)
    D, R, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, 1, 1, k, float(g["alpha"]), A, TYPE_CODE[t],
                          1, B, TYPE_CODE[t], k, float(g["beta"]), None, oracle.F32, 1,
                          tf32=(t == "f32"))
    return D[0, 0], float(g["expected_fp32"]), g


@pytest.mark.parametrize("t", ["f16", "bf16", "f32"])
def test_page_accumulation_example(t):
    got, want, _ = _golden_case("page_accumulation_example.txt", t)
    assert want == 2.25 + 2.0 ** -22
    assert got == np.float32(want)


@pytest.mark.parametrize("t", ["bf16", "f32"])
def test_page_subnormal_example(t):
    got, want, _ = _golden_case("page_subnormal_example.txt", t)
    assert want == 2.0 ** -149
    assert np.float32(got).view(np.uint32) == 1


def test_page_accumulation_example_padded_16cube():
    """The same vector embedded in a 16x16x16 FP16 GEMM (zeros elsewhere)."""
    g = load_golden("page_accumulation_example.txt")
    k = 16
    A = np.zeros((16, k))
    B = np.zeros((k, 16))
    A[0, :3] = [float(v) for v in g["a"]]
    B[:3, 0] = [float(v) for v in g["b"]]
    D, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, 16, 16, k, 1.0, _store(_colmajor(A), "f16"),
                          oracle.F16, 16, _store(_colmajor(B), "f16"), oracle.F16, k, 0.0,
                          None, oracle.F32, 16)
    assert D[0, 0] == np.float32(2.25 + 2.0 ** -22)
    assert np.count_nonzero(D) == 1


def test_numpy_float64_matmul_crosscheck():
    w = wl.custom(256, 256, 1024, "f16", "f32", alpha=1.0, beta=0.0, seed=14)
    A, B, C = wl.draw(w)
    D, R, _ = oracle_rowmajor(w, A, B, C)
    ref = A[0].astype(np.float64) @ B[0].astype(np.float64)
    assert np.max(np.abs(R - ref) / (np.abs(ref) + 1e-30)) < 1e-12
    diff = np.count_nonzero(D != ref.astype(np.float32))
    assert diff <= 1e-6 * D.size + 1


def test_degenerate_cases_follow_blas_convention():
    rng = np.random.default_rng(15)
    m, n = 9, 6
    Cv = rng.standard_normal((m, n)).astype(np.float32)
    C = _colmajor(Cv)
    # k == 0: D = beta*C, A and B are not read (passed as None)
    D, R, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, m, n, 0, 1.0, None, oracle.F16, m, None,
                          oracle.F16, 1, 0.5, C, oracle.F32, m)
    assert np.array_equal(D, (0.5 * Cv.astype(np.float64)).astype(np.float32))
    # alpha == 0: same, A and B not read
    D, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, m, n, 4, 0.0, None, oracle.F16, m, None,
                          oracle.F16, 4, -2.0, C, oracle.F32, m)
    assert np.array_equal(D, (-2.0 * Cv.astype(np.float64)).astype(np.float32))
    # beta == 0: C not read, NaN in C does not propagate
    A = _store(np.ones(m * 4), "f16")
    B = _store(np.ones(4 * n), "f16")
    Cnan = np.full(m * n, np.nan, dtype=np.float32)
    D, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, m, n, 4, 1.0, A, oracle.F16, m, B,
                          oracle.F16, 4, 0.0, Cnan, oracle.F32, m)
    assert np.all(D == 4.0)
    # empty results
    D, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, 0, n, 4, 1.0, A, oracle.F16, 1, B,
                          oracle.F16, 4, 0.0, None, oracle.F32, 1)
    assert D.size == 0


def test_fp16_output_overflow_and_specials():
    # 300 * 300 = 90000 > 65504 -> +Inf; Inf * 0 = NaN; products of opposite Inf
    A = _store(np.array([300.0, 0.0, np.inf]), "f16")          # 3 x 1
    B = _store(np.array([300.0]), "f16")                        # 1 x 1
    D, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, 3, 1, 1, 1.0, A, oracle.F16, 3, B,
                          oracle.F16, 1, 0.0, None, oracle.F16, 3)
    v = D.view(np.float16).reshape(-1)
    assert v[0] == np.inf and v[1] == 0 and v[2] == np.inf
    Bz = _store(np.array([0.0]), "f16")
    D, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, 3, 1, 1, 1.0, A, oracle.F16, 3, Bz,
                          oracle.F16, 1, 0.0, None, oracle.F32, 3)
    assert np.isnan(D[2, 0]) and D[0, 0] == 0
