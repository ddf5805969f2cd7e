"""Pins of the oracle's block-FMA model (oracle/tc_model.c), CPU only.

The model is the accumulation described in "NVIDIA Tensor Core混合精度计算原理与应用解析",
sections 2.2, 2.3 and 4.  It is pinned by that page's worked example (section 2.2.1), by
closed forms that follow from the model's definition for hand-built vectors, by
invariants, and by reduction to the exact oracle (orc_gemm) when nothing is cut.
"""
import numpy as np
import pytest

import oracle

F16, BF16 = oracle.F16, oracle.BF16


def bits(values, fmt):
    """Raw storage of exactly representable values."""
    x = np.asarray(values, dtype=np.float64)
    if fmt == F16:
        out = x.astype(np.float16)
        assert np.array_equal(out.astype(np.float64), x)
        return out.view(np.uint16)
    # BF16: the top half of the FP32 bits; exact values only
    f = x.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), x, equal_nan=True)
    u = f.view(np.uint32)
    assert np.all(u & 0xFFFF == 0), "not a BF16 value"
    return (u >> 16).astype(np.uint16)


def dot(a, b, fmt=F16, **kw):
    """Model result of one dot product (1 x 1 x k)."""
    k = len(a)
    d = oracle.dot_model(bits(a, fmt), fmt, bits(b, fmt), fmt, 1, 1, k, **kw)
    return float(d[0, 0])


# --- the page's worked example (section 2.2.1) -------------------------------------

PAGE_A = [1.5, 2.0 ** -23, 2.0 ** -24]
PAGE_B = [1.5, 1.0, 1.0]


def test_page_example_v100_accumulator():
    # 2 integer + 22 fraction bits, no extra alignment bits, block FMA of 4 (sections
    # 2.2.1, 4.1): 2^-23 and 2^-24 fall below the accumulator and the result is 2.25
    for rne in (False, True):
        assert dot(PAGE_A, PAGE_B, block=4, frac=22, norm_rne=rne) == 2.25


def test_page_example_a100_accumulator():
    # 2 + 23 + 1 bits (one extra alignment bit), block of 8, truncation inside, RNE at the
    # output (sections 2.2.1, 4.2.1): the page's answer is 2.25 + 2^-22
    assert dot(PAGE_A, PAGE_B, block=8, frac=24, norm_rne=True) == 2.25 + 2.0 ** -22


def test_page_example_inside_a_padded_16x16x16_gemm():
    rng = np.random.default_rng(0)
    A = np.zeros((16, 16))
    B = np.zeros((16, 16))
    A[0, :3] = PAGE_A
    B[:3, 0] = PAGE_B
    # other rows/columns: small integers, irrelevant to D[0, 0]
    A[1:, :] = rng.integers(-2, 3, (15, 16))
    B[:, 1:] = rng.integers(-2, 3, (16, 15))
    Ab = bits(A.T.reshape(-1), F16)          # column-major 16 x 16
    Bb = bits(B.T.reshape(-1), F16)
    D = oracle.dot_model(Ab, F16, Bb, F16, 16, 16, 16, block=8, frac=24, norm_rne=True)
    assert D[0, 0] == np.float32(2.25 + 2.0 ** -22)
    # integer entries are exact whatever the accumulator
    ref = A @ B
    assert np.array_equal(D[1:, 1:].astype(np.float64), ref[1:, 1:])


# --- closed forms of the model's definition -------------------------------------------

@pytest.mark.parametrize("frac", [22, 24, 25, 27])
def test_cancellation_window(frac):
    # [1, -1, 2^-j]: the block's largest alignment exponent is 0, so 2^-j survives the cut
    # exactly when j <= frac, and the result is then 2^-j, else 0
    for j in range(10, 40):
        got = dot([1.0, -1.0, 2.0 ** -j], [1.0, 1.0, 1.0], fmt=BF16, block=16, frac=frac)
        assert got == (2.0 ** -j if j <= frac else 0.0), (frac, j, got)


@pytest.mark.parametrize("block", [4, 8, 16])
def test_block_boundary(block):
    # [1 at 0, -1 at 1, d at p]: d is cut away inside the block of the +-1 pair and kept
    # once it starts a block of its own (the accumulator is then exactly 0)
    d = 2.0 ** -40
    for p in range(2, 40):
        a = [0.0] * 40
        a[0], a[1], a[p] = 1.0, -1.0, d
        got = dot(a, [1.0] * 40, fmt=BF16, block=block, frac=25)
        assert got == (d if p >= block else 0.0), (block, p, got)


def test_normalisation_rounding():
    # 1 + 2^-23 + 2^-24 is kept exactly (frac >= 24) and lies 1.5 ulp above 1: toward
    # zero gives 1 + 2^-23, to nearest even 1 + 2^-22; the same with signs flipped
    a, b = [1.0, 2.0 ** -23, 2.0 ** -24], [1.0, 1.0, 1.0]
    assert dot(a, b, frac=25, norm_rne=False) == 1 + 2.0 ** -23
    assert dot(a, b, frac=25, norm_rne=True) == 1 + 2.0 ** -22
    na = [-x for x in a]
    assert dot(na, b, frac=25, norm_rne=False) == -(1 + 2.0 ** -23)
    assert dot(na, b, frac=25, norm_rne=True) == -(1 + 2.0 ** -22)


def test_alignment_exponent_convention():
    # 1.5 * 1.5 = 2.25 has input exponents 0 + 0 but product exponent 1: with input sums
    # the cut is at 2^-25 and 2^-25 survives, with product exponents the cut is at 2^-24
    a, b = [1.5, -1.5, 2.0 ** -25], [1.5, 1.5, 1.0]
    assert dot(a, b, fmt=BF16, frac=25, exp_sum=True) == 2.0 ** -25
    assert dot(a, b, fmt=BF16, frac=25, exp_sum=False) == 0.0


def test_accumulator_takes_part_in_the_alignment():
    # block 1 = [1, 0, ...]; block 2 = eight products 2^-26: aligned to the accumulator
    # (exponent 0) each is cut at 2^-25 and the sum stays 1 (summed on their own they would
    # make 2^-23 and 1 + 2^-23); eight 2^-25 survive and make 1 + 2^-22
    a = [1.0] + [0.0] * 7 + [2.0 ** -26] * 8
    assert dot(a, [1.0] * 16, fmt=BF16, block=8, frac=25) == 1.0
    a = [1.0] + [0.0] * 7 + [2.0 ** -25] * 8
    assert dot(a, [1.0] * 16, fmt=BF16, block=8, frac=25) == 1 + 2.0 ** -22
    # one product per block: every 2^-26 meets the accumulator alone and is cut
    a = [1.0] + [2.0 ** -26] * 8
    assert dot(a, [1.0] * 9, fmt=BF16, block=1, frac=25) == 1.0


def test_fp32_subnormal_outputs():
    # 1.5 * 2^-150 = 0.75 * 2^-149: toward zero 0, to nearest 2^-149; 1.75 * 2^-149:
    # toward zero 2^-149, to nearest 2^-148
    a, b = [1.5 * 2.0 ** -100], [2.0 ** -50]
    assert dot(a, b, fmt=BF16, norm_rne=False) == 0.0
    assert dot(a, b, fmt=BF16, norm_rne=True) == 2.0 ** -149
    a, b = [1.75 * 2.0 ** -100], [2.0 ** -49]
    assert dot(a, b, fmt=BF16, norm_rne=False) == 2.0 ** -149
    assert dot(a, b, fmt=BF16, norm_rne=True) == 2.0 ** -148


def test_special_values():
    inf, nan = float("inf"), float("nan")
    assert dot([inf, 1.0], [1.0, 1.0], fmt=BF16) == inf
    assert np.isnan(dot([inf, -inf], [1.0, 1.0], fmt=BF16))
    assert np.isnan(dot([inf, 0.0], [0.0, 1.0], fmt=BF16))          # Inf * 0
    assert np.isnan(dot([nan, 1.0], [1.0, 1.0], fmt=BF16))
    # Inf from the first block stays in the accumulator
    assert dot([inf] + [1.0] * 20, [1.0] * 21, fmt=BF16, block=4) == inf


# --- invariants -----------------------------------------------------------------------

def _random_f16(rng, shape, lo=-14, hi=4):
    e = rng.integers(lo, hi, shape)
    m = rng.integers(0, 1024, shape)
    s = rng.integers(0, 2, shape) * 2 - 1
    return (s * np.ldexp(1.0 + m / 1024.0, e)).astype(np.float16)


def test_sign_symmetry():
    # cuts toward zero and both roundings are symmetric: model(-A, B) == -model(A, B)
    rng = np.random.default_rng(3)
    m, n, k = 8, 8, 64
    A = _random_f16(rng, (k, m))                 # column-major m x k
    B = _random_f16(rng, (n, k))                 # column-major k x n
    for rne in (False, True):
        D1 = oracle.dot_model(A.view(np.uint16), F16, B.view(np.uint16), F16, m, n, k,
                               frac=25, norm_rne=rne)
        D2 = oracle.dot_model((-A).view(np.uint16), F16, B.view(np.uint16), F16, m, n, k,
                               frac=25, norm_rne=rne)
        assert np.array_equal(D1, -D2)


def test_reduces_to_the_exact_oracle_when_nothing_is_cut():
    # one block over all of k, a 60-bit cut and round-to-nearest-even: the model is the
    # exact sum rounded once -- orc_gemm's result (inputs chosen so that its FP64 sum is
    # exact: FP16 multiples of 2^-11 in [-1, 1], k = 256)
    rng = np.random.default_rng(4)
    m, n, k = 32, 24, 256
    A = (rng.integers(-2048, 2049, (k, m)) / 2048.0).astype(np.float16)
    B = (rng.integers(-2048, 2049, (n, k)) / 2048.0).astype(np.float16)
    Dm = oracle.dot_model(A.view(np.uint16), F16, B.view(np.uint16), F16, m, n, k, block=k,
                           frac=60, norm_rne=True)
    Do, _, _ = oracle.gemm(oracle.OP_N, oracle.OP_N, m, n, k, 1.0, A.view(np.uint16), F16, m,
                           B.view(np.uint16), F16, k, 0.0, None, oracle.F32, m)
    assert np.array_equal(Dm, Do)


def test_truncation_error_stays_inside_the_bound():
    # with the cut at 25 bits and truncated blocks, every result stays within the error
    # bound the GPU parity tests use: k * 2^-23 * sum |a||b|
    rng = np.random.default_rng(5)
    m, n, k = 16, 16, 512
    A = _random_f16(rng, (k, m))
    B = _random_f16(rng, (n, k))
    D = oracle.dot_model(A.view(np.uint16), F16, B.view(np.uint16), F16, m, n, k, block=16,
                          frac=25, norm_rne=False).astype(np.float64)
    Af = A.astype(np.float64).reshape(k, m).T     # m x k
    Bf = B.astype(np.float64).reshape(n, k).T     # k x n
    exact = Af @ Bf
    bound = k * 2.0 ** -23 * (np.abs(Af) @ np.abs(Bf))
    assert np.all(np.abs(D - exact) <= bound)


def test_split_k_partials_are_added_in_fp32():
    # K = 32 in two ranges of 16: range 0 = [1, 2^-23] -> 1 + 2^-23, range 1 = [1.5 * 2^-24]
    # kept exactly on its own; their FP32 sum (nearest even) is 1 + 2^-22.  Unsplit, the
    # second block meets the accumulator 1 + 2^-23 and the truncated sum stays 1 + 2^-23.
    a = [1.0, 2.0 ** -23] + [0.0] * 14 + [1.5 * 2.0 ** -24] + [0.0] * 15
    b = [1.0] * 32
    assert dot(a, b, fmt=BF16, block=16, frac=25) == 1 + 2.0 ** -23
    assert dot(a, b, fmt=BF16, block=16, frac=25, splits=2, k_per_split=16) == 1 + 2.0 ** -22


def test_split_k_integer_data_is_exact():
    # small integers: every partial and their sum are exact, whatever the split
    rng = np.random.default_rng(6)
    m, n, k = 12, 10, 300
    A = rng.integers(-2, 3, (k, m)).astype(np.float16)
    B = rng.integers(-2, 3, (n, k)).astype(np.float16)
    ref = A.astype(np.float64).reshape(k, m).T @ B.astype(np.float64).reshape(n, k).T
    for splits, kps in ((1, 0), (2, 256), (3, 128), (5, 64)):
        D = oracle.dot_model(A.view(np.uint16), F16, B.view(np.uint16), F16, m, n, k,
                             splits=splits, k_per_split=kps)
        assert np.array_equal(D.astype(np.float64), ref), (splits, kps)


def test_split_k_rejects_empty_ranges():
    A = np.zeros(64, dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.dot_model(A, F16, A, F16, 1, 1, 64, splits=3, k_per_split=32)
