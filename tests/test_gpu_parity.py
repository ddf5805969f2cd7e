"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar (element by element): bit-exact (by value class) on integer-valued inputs
whose sums stay exact in FP32; on random inputs
    |D - ref| <= k*2^-23*(|alpha|*(|A||B|) + |beta|*|C|)  (+ one output ulp for 16-bit out)
the error model of "NVIDIA Tensor Core混合精度计算原理与应用解析" section 2.3 with
p = 23 (FP32 accumulation), against the exact oracle -- and, in addition, bit-exact
(by value class) against the oracle's block-FMA model (oracle.MODEL): for FP16, BF16
and TF32 with the parameters that page gives for its newest generation
(oracle.PAGE_MODEL: blocks of 16 FP16/BF16 or 8 TF32 products, a cut 25 bits below the
block's largest exponent, truncation); for FP8 with the parameters the feature probe
measured on this GPU (oracle.MEASURED_MODEL: one block per 32-element instruction).  Small cases are checked in full; the 8192^3,
16384x4096x4096 and 4096x4096x16384 workloads are checked on 64 seeded 128x128
output tiles (corners always included), in the launch configuration the
benchmark times.  Output buffers carry canary guard bands (before, after, and in
the ldc padding) that must stay untouched.
"""
import numpy as np
import pytest
import torch

import mixed_precision_tensor_gb300 as tcg
import oracle
from helpers import (TYPE_CODE, check_bound, decode_out, model_block, model_rowmajor,
                     oracle_rowmajor, raw, values_equal)
from mixed_precision_tensor_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N, T = tcg.TCG_OP_N, tcg.TCG_OP_T
CODE = {"f16": tcg.TCG_R_16F, "bf16": tcg.TCG_R_16BF, "f32": tcg.TCG_R_32F,
        "e4m3": tcg.TCG_R_8F_E4M3, "e5m2": tcg.TCG_R_8F_E5M2}
ESIZE = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}


@pytest.fixture(scope="module")
def handle(cuda_device):
    h = tcg.Handle()
    yield h
    h.close()


@pytest.fixture(scope="module", params=[(1, 0), (2, 256), (2, 128)],
                ids=["1sm", "2sm", "2sm-n128"])
def any_handle(cuda_device, request):
    """A handle on each kernel variant: single-SM 128x256 tiles, SM-pair 256x256 tiles and
    SM-pair 256x128 tiles (FP16/BF16 inputs; the others fall back to 256 columns)."""
    h = tcg.Handle()
    cta_group, tile_n = request.param
    tcg.check(tcg.tcg_set_kernel_options(h.h, cta_group, 0))
    tcg.check(tcg.tcg_set_tile_n(h.h, tile_n))
    yield h
    h.close()


def _to_storage(x64, t):
    if t in ("e4m3", "e5m2"):
        dt = torch.float8_e4m3fn if t == "e4m3" else torch.float8_e5m2
        return torch.from_numpy(x64.astype(np.float32)).to(dt).view(torch.uint8).numpy()
    if t == "f16":
        return x64.astype(np.float32).astype(np.float16).view(np.uint16)
    if t == "bf16":
        return torch.from_numpy(x64.astype(np.float32)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
    return x64.astype(np.float32)


def _t(a):
    """numpy -> torch without uint16 (limited in torch): raw 16-bit data as int16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a)


def _decode(raw_arr, t):
    if t == "f16":
        return raw_arr.view(np.float16).astype(np.float64)
    if t == "bf16":
        return oracle.bf16_to_f64(raw_arr)
    return raw_arr.astype(np.float64)


def _draw_values(rng, shape, dist):
    if dist == "integer":
        return rng.integers(-2, 3, shape).astype(np.float64)
    return rng.uniform(-1, 1, shape)


def _roundup(x, a):
    return max(a, (x + a - 1) // a * a)


CANARY = {"f32": np.array([0x7FC0DEAD], dtype=np.uint32).view(np.float32)[0],
          "f16": np.uint16(0x7E5A), "bf16": np.uint16(0x7FDA)}


def run_colmajor(h, transa, transb, m, n, k, alpha, beta, in_t, out_t, seed, dist,
                 extra_ld=0, batch=1, split3=False):
    """One column-major call through the C ABI on padded buffers with guard bands;
    returns (got, ref, R, absAB, Cdecoded) as column-major (m, n) blocks per batch,
    plus a flag saying whether the guard bands survived."""
    rng = np.random.default_rng(seed)
    ain = 16 // ESIZE[in_t]
    aout = 16 // ESIZE[out_t]
    a_rows, a_cols = (m, k) if transa == N else (k, m)
    b_rows, b_cols = (k, n) if transb == N else (n, k)
    lda = _roundup(a_rows, ain) + extra_ld * ain
    ldb = _roundup(b_rows, ain) + extra_ld * ain
    ldc = _roundup(m, aout) + extra_ld * aout
    sA, sB, sC = lda * a_cols, ldb * b_cols, ldc * n
    sA, sB, sC = _roundup(sA, ain), _roundup(sB, ain), _roundup(sC, aout)
    Araw = _to_storage(_draw_values(rng, batch * sA, dist), in_t)
    Braw = _to_storage(_draw_values(rng, batch * sB, dist), in_t)
    if dist == "integer":
        Cv = rng.integers(-8, 9, batch * sC).astype(np.float64)
        if out_t != "f32":
            Cv = Cv / 2.0
    else:
        Cv = rng.standard_normal(batch * sC)
    Craw = _to_storage(Cv, out_t)
    guard = 64
    canary = CANARY[out_t]
    Cbuf = np.full(batch * sC + 2 * guard, canary, dtype=Craw.dtype)
    Cbuf[guard:guard + batch * sC] = Craw
    # ldc padding rows hold canaries too (they must survive)
    view = Cbuf[guard:guard + batch * sC].reshape(batch, sC)[:, : ldc * n].reshape(batch, n, ldc)
    view[:, :, m:] = canary
    Cin = Cbuf[guard:guard + batch * sC].copy()
    dev = torch.device("cuda:0")
    dA = _t(Araw).to(dev)
    dB = _t(Braw).to(dev)
    dC = _t(Cbuf).to(dev)
    cptr = dC.data_ptr() + guard * Cbuf.itemsize
    comp = tcg.TCG_COMPUTE_32F_FAST_TF32 if in_t == "f32" else tcg.TCG_COMPUTE_32F
    if split3:
        comp = tcg.TCG_COMPUTE_32F_3XTF32
    if batch == 1:
        s = tcg.tcg_gemm_ex(h.h, transa, transb, m, n, k, alpha, dA, CODE[in_t], lda, dB,
                            CODE[in_t], ldb, beta, cptr, CODE[out_t], ldc, comp)
    else:
        s = tcg.tcg_gemm_strided_batched(h.h, transa, transb, m, n, k, alpha, dA, CODE[in_t],
                                         lda, sA, dB, CODE[in_t], ldb, sB, beta, cptr,
                                         CODE[out_t], ldc, sC, batch, comp)
    tcg.check(s, "gemm")
    tcg.check(tcg.tcg_get_device_error(h.h), "device error")
    out = dC.cpu().numpy().view(Cbuf.dtype)
    guards_ok = (np.array_equal(out[:guard].view(np.uint8), Cbuf[:guard].view(np.uint8)) and
                 np.array_equal(out[-guard:].view(np.uint8), Cbuf[-guard:].view(np.uint8)))
    body = out[guard:guard + batch * sC].reshape(batch, sC)
    pad = body[:, : ldc * n].reshape(batch, n, ldc)[:, :, m:]
    guards_ok = guards_ok and np.array_equal(pad.view(np.uint8),
                                             np.full_like(pad, canary).view(np.uint8))
    # the K ranges this call gave every tile (the model accumulates the same ranges)
    st, tm, tn, tsplits, tkps = tcg.tcg_gemm_tile_plan(h.h, m, n, k, CODE[in_t], comp,
                                                       CODE[out_t], batch)
    tcg.check(st, "tile plan")
    plan = (tm, tn, tsplits, tkps)
    results = []
    for b in range(batch):
        args = (transa, transb, m, n, k, alpha, Araw[b * sA:(b + 1) * sA], TYPE_CODE[in_t], lda,
                Braw[b * sB:(b + 1) * sB], TYPE_CODE[in_t], ldb, beta,
                Cin[b * sC:(b + 1) * sC], TYPE_CODE[out_t], ldc)
        D, R, AB = oracle.gemm(*args, tf32=(in_t == "f32" and not split3))
        # the three-product FP32 emulation is three GEMMs: not one block-FMA accumulation
        Dm = None if split3 else model_block(args, (0, m), (0, n), plan=plan, batch_entry=b,
                                             tf32=(in_t == "f32"),
                                             **oracle.MODEL[TYPE_CODE[in_t]])
        got = body[b, : ldc * n].reshape(n, ldc)[:, :m].T
        cdec = _decode(Cin[b * sC:(b + 1) * sC][: ldc * n].reshape(n, ldc)[:, :m].T, out_t)
        results.append((got, D, R, AB, cdec, Dm))
    return results, guards_ok


def _assert_results(results, k, alpha, beta, out_t, exact):
    for got, D, R, AB, cdec, Dm in results:
        g = _decode(np.ascontiguousarray(got), out_t)
        ref = _decode(np.ascontiguousarray(D), out_t)
        if exact:
            assert values_equal(g, ref), f"max |diff| {np.nanmax(np.abs(g - ref))}"
        else:
            ok, worst, idx = check_bound(g, ref, AB, cdec, k, alpha, beta, out_t)
            assert ok, f"bound exceeded: worst normalised error {worst} at {np.unravel_index(idx, g.shape)}"
        if Dm is not None:
            _assert_model_equal(g, _decode(np.ascontiguousarray(Dm), out_t))


def _assert_model_equal(g, model):
    """Bit-exact (by value class) against the block-FMA model."""
    same = (g == model) | (np.isnan(g) & np.isnan(model))
    bad = np.argwhere(~same)
    assert bad.size == 0, (f"{len(bad)} of {g.size} differ from the block-FMA model; first "
                           f"(index, gpu, model): " +
                           str([(tuple(int(x) for x in i), float(g[tuple(i)]),
                                 float(model[tuple(i)])) for i in bad[:4]]))


RAGGED = [(1, 1, 1), (7, 17, 15), (129, 255, 257), (200, 127, 1000), (257, 513, 64),
          (1000, 300, 129), (128, 256, 64), (33, 1, 300), (1, 260, 8)]


@pytest.mark.parametrize("m,n,k", RAGGED)
@pytest.mark.parametrize("in_t,out_t", [("f16", "f32"), ("f16", "f16"), ("bf16", "f32"),
                                        ("bf16", "bf16"), ("f32", "f32")])
def test_ragged_integer_bitexact(any_handle, m, n, k, in_t, out_t):
    handle = any_handle
    res, guards = run_colmajor(handle, N, N, m, n, k, 1.0, 1.0, in_t, out_t, seed=m * 7 + n + k,
                               dist="integer")
    assert guards, "guard band or ldc padding overwritten"
    _assert_results(res, k, 1.0, 1.0, out_t, exact=True)


@pytest.mark.parametrize("m,n,k", RAGGED)
@pytest.mark.parametrize("in_t,out_t", [("f16", "f32"), ("f16", "f16"), ("bf16", "f32"),
                                        ("f32", "f32")])
def test_ragged_random_within_bound(handle, m, n, k, in_t, out_t):
    res, guards = run_colmajor(handle, N, N, m, n, k, 0.75, -0.5, in_t, out_t,
                               seed=1000 + m + n * 3 + k, dist="uniform", extra_ld=1)
    assert guards
    _assert_results(res, k, 0.75, -0.5, out_t, exact=False)


@pytest.mark.parametrize("transa", [N, T])
@pytest.mark.parametrize("transb", [N, T])
@pytest.mark.parametrize("in_t", ["f16", "bf16", "f32"])
def test_all_op_combinations(any_handle, transa, transb, in_t):
    handle = any_handle
    m, n, k = 300, 520, 200
    res, guards = run_colmajor(handle, transa, transb, m, n, k, 1.0, 1.0, in_t, "f32",
                               seed=5 + transa * 2 + transb, dist="integer", extra_ld=2)
    assert guards
    _assert_results(res, k, 1.0, 1.0, "f32", exact=True)
    res, guards = run_colmajor(handle, transa, transb, m, n, k, 1.5, 0.25, in_t, "f32",
                               seed=50 + transa * 2 + transb, dist="uniform")
    assert guards
    _assert_results(res, k, 1.5, 0.25, "f32", exact=False)


# M/N multiples of 64 and K a multiple of 8: M/N-major operands take the interleaved
# (5-D tensor map) layout; K % 64 != 0 exercises its zero-filled K tail.
INTERLEAVED = [(320, 448, 200), (192, 64, 8), (640, 384, 1000), (128, 128, 72)]


@pytest.mark.parametrize("m,n,k", INTERLEAVED)
@pytest.mark.parametrize("transa", [N, T])
@pytest.mark.parametrize("transb", [N, T])
def test_interleaved_mn_layout(any_handle, m, n, k, transa, transb):
    for in_t in ("f16", "bf16", "f32"):
        res, guards = run_colmajor(any_handle, transa, transb, m, n, k, 1.0, 1.0, in_t, "f32",
                                   seed=m + n + k + transa, dist="integer")
        assert guards
        _assert_results(res, k, 1.0, 1.0, "f32", exact=True)
    res, guards = run_colmajor(any_handle, transa, transb, m, n, k, 0.5, 2.0, "f16", "f16",
                               seed=7 * m + k, dist="uniform", batch=2)
    assert guards
    _assert_results(res, k, 0.5, 2.0, "f16", exact=False)


@pytest.mark.parametrize("in_t,out_t", [("f16", "f16"), ("f16", "f32"), ("f32", "f32")])
def test_strided_batched_ragged(any_handle, in_t, out_t):
    res, guards = run_colmajor(any_handle, N, T, 100, 72, 40, 1.0, 0.5, in_t, out_t, seed=77,
                               dist="integer", batch=5)
    assert guards
    _assert_results(res, 40, 1.0, 0.5, out_t, exact=True)


SPLIT3_SHAPES = [(1, 1, 1), (129, 255, 257), (300, 520, 1000), (256, 256, 4096), (64, 900, 33)]


@pytest.mark.parametrize("m,n,k", SPLIT3_SHAPES)
@pytest.mark.parametrize("transa,transb", [(N, N), (T, N), (N, T), (T, T)])
def test_split3_tf32_recovers_fp32_accuracy(any_handle, m, n, k, transa, transb):
    """Three-product TF32 split ("NVIDIA Tensor Core混合精度计算原理与应用解析", section
    5.1) against the oracle's exact product of the FP32 inputs: within
    (k + 8)*2^-23*(|alpha||A||B| + |beta||C|), and far below plain TF32's error."""
    kw = dict(seed=31 * m + n + k + transa, dist="uniform")
    res3, guards = run_colmajor(any_handle, transa, transb, m, n, k, 0.75, -0.5, "f32", "f32",
                                split3=True, **kw)
    assert guards
    res1, _ = run_colmajor(any_handle, transa, transb, m, n, k, 0.75, -0.5, "f32", "f32",
                           **kw)
    (got3, D, R, AB, cdec, _), (got1, _, _, _, _, _) = res3[0], res1[0]
    scale = 0.75 * AB + 0.5 * np.abs(cdec)
    bound = (k + 8) * 2.0 ** -23 * scale
    err3 = np.abs(got3.astype(np.float64) - R)
    err1 = np.abs(got1.astype(np.float64) - R)
    assert np.all(err3 <= bound), f"worst {np.max(err3 / np.maximum(bound, 1e-300))}"
    # plain TF32 (one product of rounded inputs) carries the inputs' 2^-11 rounding; the
    # split leaves only the FP32 accumulation error, which grows with k: it must still be
    # clearly better (measured ~20x at k = 4096, more for small k)
    if k >= 8:
        assert np.max(err1 / np.maximum(scale, 1e-30)) > 8 * np.max(err3 / np.maximum(scale, 1e-30))


def test_split3_batched_and_integer_exact(any_handle):
    res, guards = run_colmajor(any_handle, N, T, 100, 72, 40, 1.0, 0.5, "f32", "f32", seed=91,
                               dist="integer", batch=3, split3=True)
    assert guards
    for got, D, R, AB, cdec, _ in res:
        assert values_equal(got.astype(np.float64), R)


FP8_SHAPES = [(1, 1, 1), (7, 17, 15), (129, 255, 257), (256, 384, 1000), (1000, 300, 129)]


@pytest.mark.parametrize("m,n,k", FP8_SHAPES)
@pytest.mark.parametrize("in_t", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out_t", ["f32", "f16", "bf16"])
def test_fp8_ragged(any_handle, m, n, k, in_t, out_t):
    """FP8 (E4M3 / E5M2) inputs, exact products, FP32 accumulation: bit-exact on integer
    data, within the bound on random data."""
    res, guards = run_colmajor(any_handle, N, N, m, n, k, 1.0, 1.0, in_t, out_t,
                               seed=m + 3 * n + k, dist="integer")
    assert guards
    _assert_results(res, k, 1.0, 1.0, out_t, exact=True)
    res, guards = run_colmajor(any_handle, N, N, m, n, k, 0.5, -1.0, in_t, out_t,
                               seed=5 + m + n + k, dist="uniform", extra_ld=1)
    assert guards
    _assert_results(res, k, 0.5, -1.0, out_t, exact=False)


@pytest.mark.parametrize("m,n,k", [(256, 512, 320), (384, 128, 64), (300, 520, 200)])
@pytest.mark.parametrize("transa,transb", [(N, N), (T, N), (N, T), (T, T)])
@pytest.mark.parametrize("in_t", ["e4m3", "e5m2"])
def test_fp8_op_combinations(any_handle, m, n, k, transa, transb, in_t):
    res, guards = run_colmajor(any_handle, transa, transb, m, n, k, 1.0, 1.0, in_t, "f32",
                               seed=11 + m + transa + 2 * transb, dist="integer", batch=2)
    assert guards
    _assert_results(res, k, 1.0, 1.0, "f32", exact=True)


def test_degenerate_cases(handle):
    # k == 0 and alpha == 0: D = beta*C, A/B not read (NULL)
    for k, alpha in ((0, 1.0), (64, 0.0)):
        m, n = 70, 40
        C = torch.randn(n, 72, device="cuda")        # column-major m x n, ldc = 72
        want = (-1.5 * C.double()).float()
        s = tcg.tcg_gemm_ex(handle.h, N, N, m, n, k, alpha, None, tcg.TCG_R_16F, 72, None,
                            tcg.TCG_R_16F, 64, -1.5, C, tcg.TCG_R_32F, 72, tcg.TCG_COMPUTE_32F)
        tcg.check(s)
        torch.cuda.synchronize()
        assert torch.equal(C[:, :m], want[:, :m])
    # beta == 0: NaN in C does not propagate
    A = torch.ones(64, 64, dtype=torch.float16, device="cuda")
    B = torch.ones(64, 64, dtype=torch.float16, device="cuda")
    C = torch.full((64, 64), float("nan"), device="cuda")
    tcg.gemm_rowmajor(handle, A, B, C, alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    assert torch.all(C == 64.0)


def test_page_vectors_on_gpu(handle):
    """The accumulation vector of section 2.2.1 and the subnormal vector of section
    2.2.3 ("NVIDIA Tensor Core混合精度计算原理与应用解析"), padded to 16x16x16.  The
    oracle value is pinned on CPU; the hardware value is recorded and must lie
    within the bound (either truncating or rounding accumulation is acceptable)."""
    A = torch.zeros(16, 16, dtype=torch.float16)
    B = torch.zeros(16, 16, dtype=torch.float16)
    A[0, :3] = torch.tensor([1.5, 2.0 ** -23, 2.0 ** -24], dtype=torch.float16)
    B[:3, 0] = torch.tensor([1.5, 1.0, 1.0], dtype=torch.float16)
    C = torch.zeros(16, 16, device="cuda")
    tcg.gemm_rowmajor(handle, A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    v = float(C[0, 0])
    model = float(oracle.dot_model(A.T.contiguous().numpy().view(np.uint16), oracle.F16,
                                   B.T.contiguous().numpy().view(np.uint16), oracle.F16, 16, 16,
                                   16, **oracle.PAGE_MODEL[oracle.F16])[0, 0])
    assert v == model          # 2.25: 3*2^-24 cut away when the sum is truncated into FP32
    print(f"accumulation vector: GPU {v!r} (model {model!r}; exact-sum oracle 2.25 + 2^-22)")
    A = torch.zeros(16, 16, dtype=torch.bfloat16)
    B = torch.zeros(16, 16, dtype=torch.bfloat16)
    A[0, :2] = torch.tensor([127 * 2.0 ** -78, 2.0 ** -78], dtype=torch.float64).to(torch.bfloat16)
    B[:2, 0] = torch.tensor([2.0 ** -78, 2.0 ** -79], dtype=torch.float64).to(torch.bfloat16)
    C = torch.zeros(16, 16, device="cuda")
    tcg.gemm_rowmajor(handle, A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    v = float(C[0, 0])
    model = float(oracle.dot_model(A.T.contiguous().view(torch.int16).numpy().view(np.uint16),
                                   oracle.BF16,
                                   B.T.contiguous().view(torch.int16).numpy().view(np.uint16),
                                   oracle.BF16, 16, 16, 16, **oracle.PAGE_MODEL[oracle.BF16])[0, 0])
    print(f"subnormal vector: GPU {v!r} (model {model!r}; exact-sum oracle 2^-149)")
    assert v == model          # 2^-149 - 2^-157 truncated to the FP32 subnormal grid: 0


# ------------------------------------------------------------ split-K
SPLITK_CASES = [
    # (m, n, k, in, out, alpha, beta, batch, forced splits)
    (256, 256, 65536, "f16", "f32", 1.0, 0.0, 1, 0),
    (100, 300, 20000, "bf16", "bf16", 0.5, 1.0, 1, 0),
    (257, 129, 10000, "f32", "f32", 1.0, 0.0, 1, 0),
    (128, 128, 16384, "f16", "f16", 1.0, 0.5, 3, 0),
    (256, 256, 32768, "e4m3", "f32", 1.0, 0.0, 1, 0),
    (300, 700, 5000, "f16", "f32", -1.0, 0.25, 1, 3),
    (64, 64, 1000, "f16", "f32", 1.0, 0.0, 1, 64),
]


@pytest.mark.timeout(900)
@pytest.mark.parametrize("m,n,k,in_t,out_t,alpha,beta,batch,forced", SPLITK_CASES)
def test_split_k(cuda_device, m, n, k, in_t, out_t, alpha, beta, batch, forced):
    """Few output tiles, long K: the K range is split (automatically, or forced), the
    partial sums reduced in range order.  Within the bound of the exact oracle and bit-exact
    against the block-FMA model with the same split."""
    h = tcg.Handle()
    tcg.check(tcg.tcg_set_split_k(h.h, forced))
    comp = tcg.TCG_COMPUTE_32F_FAST_TF32 if in_t == "f32" else tcg.TCG_COMPUTE_32F
    st, splits, kps = tcg.tcg_gemm_split_k(h.h, m, n, k, CODE[in_t], comp, batch)
    assert st == 0 and splits > 1, (splits, kps)
    for dist in ("uniform", "integer"):
        res, guards = run_colmajor(h, N, N, m, n, k, alpha, beta, in_t, out_t,
                                   seed=m + n + k + batch, dist=dist, batch=batch)
        assert guards
        _assert_results(res, k, alpha, beta, out_t, exact=(dist == "integer"))
    h.close()


# ------------------------------------------------------------ tail split
TAIL_CASES = [
    # row-major m x n x k, in, out, alpha, beta: 77 output tiles of the column-major call
    # (1792 x 2816) on 76 SM pairs, long K -> the one tile of the partial second wave (the
    # corner tile, last in raster order) is cut in four K ranges
    (2816, 1792, 20480, "f16", "f32", 1.0, 0.0),
    (2816, 1792, 20480, "bf16", "f32", 0.5, 1.0),
]


@pytest.mark.timeout(900)
@pytest.mark.parametrize("m,n,k,in_t,out_t,alpha,beta", TAIL_CASES)
def test_tail_split(handle, m, n, k, in_t, out_t, alpha, beta):
    """Tail tiles cut along K, partial sums reduced by a second kernel: within the bound of
    the exact oracle and bit-exact against the block-FMA model with the same per-tile K
    ranges (sampled tiles, corners included)."""
    w = wl.custom(m, n, k, in_t, out_t, alpha, beta, 1, seed=m + k)
    plan = _plan(handle, w)
    assert (plan["plan"][2] > 1).any(), "expected split tail tiles"
    A, B, C = wl.draw(w)
    out = _run_workload(handle, w, A, B, C)
    _check_sampled(w, A, B, C, out, exact=False, count=12, model_tiles=6, **plan)
    wi = wl.with_dist(w, "integer")
    A, B, C = wl.draw(wi)
    out = _run_workload(handle, wi, A, B, C)
    _check_sampled(wi, A, B, C, out, exact=True, count=6)


# ------------------------------------------------------------ the five workloads
def _device_inputs(w, A, B, C):
    dev = torch.device("cuda:0")
    dA = _t(A if w.batch > 1 else A[0]).to(dev)
    dB = _t(B if w.batch > 1 else B[0]).to(dev)
    if w.in_type == "bf16":
        dA, dB = dA.view(torch.bfloat16), dB.view(torch.bfloat16)
    if w.in_type in ("e4m3", "e5m2"):
        f8 = torch.float8_e4m3fn if w.in_type == "e4m3" else torch.float8_e5m2
        dA, dB = dA.view(f8), dB.view(f8)
    shape = (w.batch, w.m, w.n) if w.batch > 1 else (w.m, w.n)
    odt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.out_type]
    if C is not None:
        dC = _t(C if w.batch > 1 else C[0]).to(dev)
        if w.out_type == "bf16":
            dC = dC.view(torch.bfloat16)
    else:
        dC = torch.empty(shape, dtype=odt, device=dev)
    return dA, dB, dC


def _run_workload(handle, w, A, B, C):
    dA, dB, dC = _device_inputs(w, A, B, C)
    tcg.gemm_rowmajor(handle, dA, dB, dC, alpha=w.alpha, beta=w.beta, tf32=w.in_type == "f32")
    tcg.check(tcg.tcg_get_device_error(handle.h), "device error")
    out = dC.cpu()
    if w.out_type == "bf16":
        out = out.view(torch.int16).numpy().view(np.uint16)
    else:
        out = out.numpy()
    return out if w.batch > 1 else out[None]


def _plan(handle, w):
    """Per-tile K ranges of the column-major call the workload makes."""
    comp = tcg.TCG_COMPUTE_32F_FAST_TF32 if w.in_type == "f32" else tcg.TCG_COMPUTE_32F
    st, tm, tn, splits, kps = tcg.tcg_gemm_tile_plan(handle.h, w.n, w.m, w.k, CODE[w.in_type],
                                                     comp, CODE[w.out_type], w.batch)
    tcg.check(st, "tile plan")
    return dict(plan=(tm, tn, splits, kps))


def _check_full(w, A, B, C, out, exact, plan=None):
    for b in range(w.batch):
        D, R, AB = oracle_rowmajor(w, A, B, C, b=b)
        g = decode_out(raw(out[b]), w.out_type)
        ref = decode_out(raw(D), w.out_type)
        cdec = decode_out(raw(C[b]), w.out_type) if C is not None else None
        if exact:
            assert values_equal(g, ref), f"batch {b}: not bit-exact"
        else:
            ok, worst, idx = check_bound(g, ref, AB, cdec, w.k, w.alpha, w.beta, w.out_type)
            assert ok, f"batch {b}: worst normalised error {worst}"
            Dm = model_rowmajor(w, A, B, C, b=b, plan=plan)
            _assert_model_equal(g, decode_out(raw(Dm), w.out_type))


def _check_sampled(w, A, B, C, out, exact, count=64, model_tiles=8, plan=None):
    tiles = wl.sample_tiles(w.m, w.n, count=count, tile=128, seed=w.seed)
    assert len(tiles) == min(count, (-(-w.m // 128)) * (-(-w.n // 128)))
    worst_all = 0.0
    for (i0, i1, j0, j1) in tiles:
        D, R, AB = oracle_rowmajor(w, A, B, C, rows=(i0, i1), cols=(j0, j1))
        g = decode_out(raw(np.ascontiguousarray(out[0][i0:i1, j0:j1])), w.out_type)
        ref = decode_out(raw(D), w.out_type)
        cdec = (decode_out(raw(np.ascontiguousarray(C[0][i0:i1, j0:j1])), w.out_type)
                if C is not None else None)
        if exact:
            assert values_equal(g, ref), f"tile {(i0, j0)} not bit-exact"
        else:
            ok, worst, idx = check_bound(g, ref, AB, cdec, w.k, w.alpha, w.beta, w.out_type)
            assert ok, f"tile {(i0, j0)}: worst normalised error {worst}"
            worst_all = max(worst_all, worst)
    if not exact:
        # bit-exact against the block-FMA model on the first model_tiles tiles (the four
        # corners come first)
        for (i0, i1, j0, j1) in tiles[:model_tiles]:
            g = decode_out(raw(np.ascontiguousarray(out[0][i0:i1, j0:j1])), w.out_type)
            Dm = model_rowmajor(w, A, B, C, rows=(i0, i1), cols=(j0, j1), plan=plan)
            _assert_model_equal(g, decode_out(raw(np.ascontiguousarray(Dm)), w.out_type))
    return worst_all


SMALL = ["fp16_gemm_256", "fp16_batched_512x256"]
LARGE = ["fp16_gemm_8192", "bf16_proj_16384x4096x4096", "tf32_gemm_4096x4096x16384"]


@pytest.mark.parametrize("name", SMALL)
def test_small_workload_full_random(handle, name):
    w = wl.WORKLOADS[name]
    A, B, C = wl.draw(w)
    out = _run_workload(handle, w, A, B, C)
    _check_full(w, A, B, C, out, exact=False, **_plan(handle, w))


@pytest.mark.parametrize("name", SMALL)
def test_small_workload_full_integer(handle, name):
    w = wl.with_dist(wl.WORKLOADS[name], "integer")
    A, B, C = wl.draw(w)
    out = _run_workload(handle, w, A, B, C)
    _check_full(w, A, B, C, out, exact=True)


@pytest.mark.timeout(900)
@pytest.mark.parametrize("name", LARGE)
def test_large_workload_sampled_random(handle, name):
    w = wl.WORKLOADS[name]
    A, B, C = wl.draw(w)
    out = _run_workload(handle, w, A, B, C)
    worst = _check_sampled(w, A, B, C, out, exact=False, **_plan(handle, w))
    print(f"{name}: worst normalised error over 64 tiles = {worst:.3e}")


@pytest.mark.timeout(900)
@pytest.mark.parametrize("name", LARGE)
def test_large_workload_sampled_integer(handle, name):
    w = wl.with_dist(wl.WORKLOADS[name], "integer")
    A, B, C = wl.draw(w)
    out = _run_workload(handle, w, A, B, C)
    # the 64 seeded tiles of the random-input check, the four corners among them
    _check_sampled(w, A, B, C, out, exact=True, count=64)


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32], ids=["f16", "tf32"])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_timeout_is_reported_not_hung(cuda_device, cta_group, dtype):
    """A bounded wait that runs out (a stage nobody fills) ends the kernel with a
    TIMEOUT status in the error word; the context stays usable afterwards.  With TF32
    inputs the wait that runs out is the converter warps' (the raw stage never lands)."""
    h = tcg.Handle()
    tcg.check(tcg.tcg_set_kernel_options(h.h, cta_group, 0))
    A = torch.ones(256, 256, dtype=dtype, device="cuda")
    B = torch.ones(256, 256, dtype=dtype, device="cuda")
    C = torch.zeros(256, 256, device="cuda")
    tf32 = dtype == torch.float32
    tcg.check(tcg.tcg_set_debug(h.h, 200_000_000, 1))          # 0.2 s, skip one load
    tcg.gemm_rowmajor(h, A, B, C, tf32=tf32)
    st = tcg.tcg_get_device_error(h.h)
    assert st == tcg.TCG_STATUS_TIMEOUT
    assert tcg.tcg_last_device_error_bits(h.h) != 0
    tcg.check(tcg.tcg_set_debug(h.h, 0, 0))
    tcg.gemm_rowmajor(h, A, B, C, tf32=tf32)
    assert tcg.tcg_get_device_error(h.h) == tcg.TCG_STATUS_SUCCESS
    torch.cuda.synchronize()
    assert torch.all(C == 256.0)
    h.close()


# --- seeded random configurations -----------------------------------------------------

def _fuzz_cases(count=160, seed=20261202):
    """Random (shape, ops, types, alpha, beta, batch, ld padding) combinations, drawn once
    from a fixed seed so that a failure names a reproducible case."""
    rng = np.random.default_rng(seed)
    outs = {"f16": ["f32", "f16"], "bf16": ["f32", "bf16"], "f32": ["f32"],
            "e4m3": ["f32", "f16", "bf16"], "e5m2": ["f32", "f16", "bf16"]}
    cases = []
    for i in range(count):
        in_t = str(rng.choice(["f16", "bf16", "f32", "e4m3", "e5m2"]))
        out_t = str(rng.choice(outs[in_t]))
        m, n = (int(x) for x in rng.integers(1, 420, 2))
        k = int(rng.integers(1, 900))
        transa, transb = (int(x) for x in rng.integers(0, 2, 2))
        alpha = float(rng.choice([1.0, 0.5, -2.0]))
        beta = float(rng.choice([0.0, 1.0, 0.25]))
        batch = int(rng.choice([1, 1, 3]))
        extra_ld = int(rng.integers(0, 2))
        cases.append((i, m, n, k, transa, transb, in_t, out_t, alpha, beta, batch, extra_ld))
    return cases


def test_encoder_refusal_is_reported(cuda_device):
    """A tensor map the driver refuses is a host-side failure: EXECUTION_FAILED, nothing
    launched, the handle still usable.  The refusal is real, not injected: lda = 2^40
    elements is a 2^41-byte stride, beyond the encoder's 2^40-byte limit.  With k = 1 the
    kernel would read column 0 of A only (K past 1 is zero-filled, never fetched), so the
    call stays in bounds even if a map were built."""
    h = tcg.Handle()
    F16, F32, C32 = tcg.TCG_R_16F, tcg.TCG_R_32F, tcg.TCG_COMPUTE_32F
    m, n = 64, 64
    A = torch.ones(m, dtype=torch.float16, device="cuda")            # column 0 only
    B = torch.ones(n, 8, dtype=torch.float16, device="cuda")         # k x n, ldb = 8
    C = torch.zeros(n, m, device="cuda")
    before = tcg.tcg_launch_count(h.h)
    st = tcg.tcg_gemm_ex(h.h, N, N, m, n, 1, 1.0, A, F16, 1 << 40, B, F16, 8, 0.0, C, F32, m,
                         C32)
    assert st == tcg.TCG_STATUS_EXECUTION_FAILED, tcg.tcg_status_string(st)
    assert tcg.tcg_launch_count(h.h) == before
    assert tcg.tcg_get_device_error(h.h) == tcg.TCG_STATUS_SUCCESS
    tcg.check(tcg.tcg_gemm_ex(h.h, N, N, m, n, 1, 1.0, A, F16, m, B, F16, 8, 0.0, C, F32, m,
                              C32))
    tcg.check(tcg.tcg_get_device_error(h.h))
    torch.cuda.synchronize()
    assert torch.all(C == 1.0)
    h.close()


@pytest.mark.parametrize("case", _fuzz_cases(), ids=lambda c: f"fuzz{c[0]}")
def test_seeded_random_configurations(any_handle, case):
    i, m, n, k, transa, transb, in_t, out_t, alpha, beta, batch, extra_ld = case
    res, guards_ok = run_colmajor(any_handle, transa, transb, m, n, k, alpha, beta, in_t,
                                  out_t, seed=5000 + i, dist="uniform", extra_ld=extra_ld,
                                  batch=batch)
    assert guards_ok, "guard band or ldc padding written"
    _assert_results(res, k, alpha, beta, out_t, exact=False)


def test_tile_width_rule(cuda_device):
    """Narrow (256 x 128) tiles exactly where the rule says: FP16/BF16 inputs on SM pairs,
    256-wide tiles filling at most half of the pairs, no K split at either width."""
    h = tcg.Handle()
    F16, F32, E4M3 = tcg.TCG_R_16F, tcg.TCG_R_32F, tcg.TCG_R_8F_E4M3
    C32, TF = tcg.TCG_COMPUTE_32F, tcg.TCG_COMPUTE_32F_FAST_TF32
    width = lambda m, n, k, at=F16, comp=C32, batch=1: tcg.tcg_gemm_tile_plan(
        h.h, m, n, k, at, comp, F32, batch)[2]
    assert width(256, 256, 256) == 128                 # one tile: narrow
    assert width(512, 512, 512) == 128
    assert width(8192, 8192, 64) == 256                # 1024 tiles: wide
    assert width(256, 256, 256, batch=512) == 256      # the batched shape: wide
    assert width(256, 256, 65536) == 256               # K is split: wide
    assert width(256, 256, 256, at=E4M3) == 256        # no narrow FP8 variant
    assert width(256, 256, 256, at=F32, comp=TF) == 256
    tcg.check(tcg.tcg_set_tile_n(h.h, 256))
    assert width(256, 256, 256) == 256                 # forced
    tcg.check(tcg.tcg_set_tile_n(h.h, 128))
    assert width(8192, 8192, 64) == 128
    tcg.check(tcg.tcg_set_kernel_options(h.h, 1, 0))
    assert width(256, 256, 256) == 256                 # single-CTA kernel: wide only
    h.close()


def _tie_patterns(rng, n):
    """FP32 values whose low 13 bits sit at, just below or just above the TF32 rounding
    tie (0x1000), with an odd or even last kept bit, over finite exponents (subnormals
    included); none rounds past the largest finite value."""
    sign = rng.integers(0, 2, n).astype(np.uint32) << 31
    expo = rng.integers(0, 254, n).astype(np.uint32) << 23          # 0: subnormal
    keep = rng.integers(0, 1 << 10, n).astype(np.uint32) << 13       # kept mantissa bits
    low = rng.choice(np.array([0x1000, 0x0FFF, 0x1001, 0x0000, 0x1FFF, 0x0001],
                              dtype=np.uint32), n)
    return (sign | expo | keep | low).view(np.float32)


@pytest.mark.parametrize("transa,transb", [(N, N), (T, N), (N, T), (T, T)])
def test_tf32_input_rounding_is_nearest_even(handle, transa, transb):
    """FP32 inputs reach the tensor core rounded to TF32 to nearest, ties to even (not
    cut): with the other operand an identity, D is the rounded input itself, bit for bit
    against the oracle's TF32 rounding (pinned exhaustively on the CPU).  Ties with an
    odd and an even last kept bit, values just below and above a tie, and subnormals;
    both operands, every op combination, ragged M/N/K."""
    rng = np.random.default_rng(77 + 2 * transa + transb)
    m, k = 200, 72
    dev = torch.device("cuda:0")
    for side in ("A", "B"):
        vals = _tie_patterns(rng, m * k).reshape(m, k)             # the operand's m x k values
        eye = np.eye(k, dtype=np.float32)
        if side == "A":                 # D (m x k) = vals (m x k) * I (k x k)
            M, Nn, Aop, Bop = m, k, vals, eye
        else:                           # D (k x m) = I (k x k) * vals^T (k x m)
            M, Nn, Aop, Bop = k, m, eye, vals.T.copy()
        Acol = Aop.T.copy() if transa == N else Aop.copy()          # column-major storage
        Bcol = Bop.T.copy() if transb == N else Bop.copy()
        lda = M if transa == N else k
        ldb = k if transb == N else Nn
        dA, dB = torch.from_numpy(Acol.reshape(-1)).to(dev), torch.from_numpy(Bcol.reshape(-1)).to(dev)
        C = torch.zeros(Nn * M, device=dev)
        tcg.check(tcg.tcg_gemm_ex(handle.h, transa, transb, M, Nn, k, 1.0, dA, tcg.TCG_R_32F, lda,
                                  dB, tcg.TCG_R_32F, ldb, 0.0, C, tcg.TCG_R_32F, M,
                                  tcg.TCG_COMPUTE_32F_FAST_TF32))
        tcg.check(tcg.tcg_get_device_error(handle.h))
        got = C.cpu().numpy().reshape(Nn, M).T                       # (M, Nn)
        want = oracle.tf32_round_bits(vals.view(np.uint32)).view(np.float32)
        if side == "B":
            want = want.T
        cut = (vals.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
        assert values_equal(got, want), f"operand {side}: not RNE-rounded"
        # the data does tell nearest-even from a plain cut
        assert not values_equal(cut if side == "A" else cut.T, want)


# ------------------------------------------------------------ extreme shapes
EXTREME = [
    # row-major m x n x k, batch, in, out (every leading dimension a multiple of 16 bytes):
    # 100,000 tiny products (work units past 65535, ragged 8 x 8 tiles), one row of dot
    # products of length 2^20 (one tile, K split in 64 ranges) and of 2^18 in TF32, a tall
    # and skinny product (2^20 rows, 8 columns: 4096 tiles with ragged N), and a wide one
    # (one row, 2^20 columns, FP8)
    (8, 8, 8, 100_000, "f16", "f32"),
    (1, 8, 1 << 20, 1, "bf16", "f32"),
    (1 << 20, 8, 16, 1, "f16", "f16"),
    (1, 1 << 20, 16, 1, "e4m3", "f32"),
    (1, 8, 1 << 18, 1, "f32", "f32"),
]


@pytest.mark.timeout(900)
@pytest.mark.parametrize("m,n,k,batch,in_t,out_t", EXTREME)
def test_extreme_shapes_integer_exact(handle, m, n, k, batch, in_t, out_t):
    """Shapes at the edges of the tile scheduler and the split plans, on integer inputs whose
    sums are exact: the whole result equals numpy's int64 product (a library routine),
    and sampled entries equal the exact oracle's."""
    rng = np.random.default_rng(m * 7 + n * 3 + k + batch)
    lo, hi = (-2, 3) if k <= 1 << 12 else (-1, 2)       # |sum| stays below 2^24 (and 2^11 for FP16 out)
    A = rng.integers(lo, hi, (batch, m, k)).astype(np.float64)
    B = rng.integers(lo, hi, (batch, k, n)).astype(np.float64)
    want = np.einsum("bik,bkj->bij", A.astype(np.int64), B.astype(np.int64))
    w = wl.custom(m, n, k, in_t, out_t, 1.0, 0.0, batch)
    As = _to_storage(A.reshape(-1), in_t).reshape(batch, m, k)
    Bs = _to_storage(B.reshape(-1), in_t).reshape(batch, k, n)
    if in_t == "f16":
        As, Bs = As.view(np.float16), Bs.view(np.float16)
    out = _run_workload(handle, w, As, Bs, None)
    got = decode_out(raw(np.ascontiguousarray(out)), out_t).reshape(batch, m, n)
    assert np.array_equal(got, want.astype(np.float64)), "not the exact integer product"
    # the exact oracle on a few entries (first and last batch entry, corner blocks)
    for b in sorted({0, batch - 1}):
        rows = (0, min(m, 64)) if m <= 128 else (m - 64, m)
        cols = (0, min(n, 64))
        D, _, _ = oracle_rowmajor(w, As, Bs, None, b=b, rows=rows, cols=cols)
        ref = decode_out(raw(D), out_t)
        assert values_equal(got[b, rows[0]:rows[1], cols[0]:cols[1]], ref)
