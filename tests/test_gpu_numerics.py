"""The tensor core's numeric features on this GPU (probe) and the block-FMA model's
agreement with it on random inputs.

"NVIDIA Tensor Core混合精度计算原理与应用解析", section 3: feature-detection vectors (GNFT,
section 3.1) fix the parameters of a model of the hardware's accumulation, and random
inputs (ISSM, section 3.2: normal and uniform samples plus directed special cases) check
the model against the hardware; on disagreement the model is refined (section 3.3).

Here the parameters come from this GPU (the probe), so agreement validates the model.
The GEMM's parity tests (test_gpu_parity.py) use oracle.MODEL, not these: for FP16, BF16
and TF32 the parameters the page states for its newest generation (oracle.PAGE_MODEL),
which test_probe_agrees_with_the_page_parameters checks against the probe; for FP8 the
parameters this probe measured (oracle.MEASURED_MODEL: the pages fix none for this GPU).
"""
import numpy as np
import pytest
import torch

import mixed_precision_tensor_gb300 as tcg
import oracle
from mixed_precision_tensor_gb300 import numerics

pytestmark = pytest.mark.gpu

KINDS = list(numerics.FORMATS)
ORACLE_TYPE = {"f16": oracle.F16, "bf16": oracle.BF16, "tf32": oracle.F32, "e4m3": oracle.F8E4M3,
               "e5m2": oracle.F8E5M2}


@pytest.fixture(scope="module")
def features(cuda_device):
    return numerics.probe(tcg.Handle())


def test_probe_determines_every_feature(features):
    for kind, f in features.items():
        assert not f.notes, (kind, f.notes)
        assert f.block is not None and f.frac_bits is not None, (kind, f)
        assert f.exponent is not None and f.accumulator_aligned is not None, (kind, f)
        assert f.normalisation is not None and f.cut is not None, (kind, f)
        assert f.subnormal_inputs is not None and f.specials_ieee is not None, (kind, f)
        assert f.model_parameters() is not None, (kind, f)


def test_probe_agrees_with_the_page_parameters(features):
    # FP16, BF16, TF32: the page's newest-generation parameters (sections 2.2.1, 2.2.2,
    # 2.3, 4.1) against what the probe measures on this GPU.
    for kind, f in features.items():
        if ORACLE_TYPE[kind] in oracle.PAGE_MODEL:
            assert f.model_parameters() == oracle.PAGE_MODEL[ORACLE_TYPE[kind]], (kind, f)


def test_probe_reproduces_the_recorded_fp8_parameters(features):
    # FP8: the pages fix no parameters for this GPU (section 4.3.2 describes H100's
    # grouping), so oracle.MEASURED_MODEL records what this probe measured; this re-measures
    # them, so a GPU that accumulates FP8 differently fails here before the parity tests.
    for kind, f in features.items():
        if ORACLE_TYPE[kind] in oracle.MEASURED_MODEL:
            assert f.model_parameters() == oracle.MEASURED_MODEL[ORACLE_TYPE[kind]], (kind, f)


def test_probe_matches_the_page_vectors(features):
    # The page's accumulator example (section 2.2.1) through the library on this GPU: the
    # result is 2.25 or 2.25 + 2^-22 depending on the window and the normalisation; the
    # probe's features must predict which.
    f = numerics.FORMATS["f16"]
    run = numerics._Runner(tcg.Handle(), f, torch.device("cuda:0")).run
    got = run([[(1.5, 1.5), (2.0 ** -23, 1.0), (2.0 ** -24, 1.0)]], f.k_instr)[0]
    ft = features["f16"]
    keeps_both = ft.frac_bits >= 24
    want = 2.25 + 2.0 ** -22 if (keeps_both and ft.normalisation == "nearest-even") else 2.25
    assert got == want


# --- ISSM: random and directed inputs, GPU against the model ---------------------------

def _cast(x64, kind):
    """float64 values -> device tensor of the kind's storage type (RNE casts)."""
    dt = numerics.FORMATS[kind].dtype
    return torch.from_numpy(x64.astype(np.float32)).to(dt)


def _raw(t, kind):
    """Host raw storage of a tensor for the oracle."""
    t = t.cpu().contiguous()
    if kind in ("f16", "bf16"):
        return t.view(torch.int16).numpy().view(np.uint16)
    if kind in ("e4m3", "e5m2"):
        return t.view(torch.uint8).numpy()
    return t.numpy()


def _draw(kind, dist, shape, rng):
    f = numerics.FORMATS[kind]
    if dist == "normal":
        return rng.standard_normal(shape)
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, shape)
    lo, hi = max(f.emin, -50), min(f.emax, 50)
    sign = rng.integers(0, 2, shape) * 2 - 1
    mant = 1.0 + rng.integers(0, 2 ** f.mbits, shape) / 2.0 ** f.mbits
    if dist == "wide":               # every exponent of the format (BF16/TF32: +-50)
        return sign * np.ldexp(mant, rng.integers(lo, hi, shape))
    if dist == "subnormal":          # half subnormal inputs, half small normals
        sub = rng.integers(1, 2 ** f.mbits, shape) * 2.0 ** (f.emin - f.mbits)
        nrm = np.ldexp(mant, rng.integers(f.emin, f.emin + 4, shape))
        return sign * np.where(rng.random(shape) < 0.5, sub, nrm)
    raise ValueError(dist)


def _case(kind, dist, m, n, k, seed):
    """Inputs (column-major A m x k, B k x n) for one ISSM case, as device tensors."""
    rng = np.random.default_rng(seed)
    A = _draw(kind, dist if dist != "cancel" else "wide", (k, m), rng)   # A^T row-major
    if dist == "subnormal":
        f = numerics.FORMATS[kind]
        # B scales the subnormal products into FP32's normal and subnormal range
        B = np.ldexp(1.0 + rng.integers(0, 2 ** f.mbits, (n, k)) / 2.0 ** f.mbits,
                     rng.integers(max(f.emax - 10, 0), f.emax, (n, k)))
    else:
        B = _draw(kind, dist if dist != "cancel" else "wide", (n, k), rng)
    if dist == "cancel":
        # every odd product cancels the even one before it, except where a perturbation
        # of one input by a few units leaves a residual far below the pair
        A[1::2, :] = -A[0::2, :]
        B[:, 1::2] = B[:, 0::2]
        f = numerics.FORMATS[kind]
        pert = rng.random(A[1::2, :].shape) < 0.25
        A[1::2, :] = np.where(pert, A[1::2, :] * (1 + 2.0 ** -f.mbits), A[1::2, :])
    return _cast(A, kind), _cast(B, kind)


DISTS = ["normal", "uniform", "wide", "cancel", "subnormal"]


@pytest.mark.timeout(600)
@pytest.mark.parametrize("dist", DISTS)
@pytest.mark.parametrize("kind", KINDS)
def test_issm_model_agreement(features, kind, dist):
    params = features[kind].model_parameters()
    assert params is not None
    f = numerics.FORMATS[kind]
    m = n = 128
    k = 8 * f.k_instr
    seed = 1000 + 17 * KINDS.index(kind) + DISTS.index(dist)
    At, Bt = _case(kind, dist, m, n, k, seed)
    D = torch.zeros((n, m), dtype=torch.float32, device="cuda:0")      # column-major m x n
    h = tcg.Handle()
    tcg.check(tcg.tcg_set_split_k(h.h, 1))        # one accumulation per output, no K split
    tcg.check(tcg.tcg_gemm_ex(h.h, tcg.TCG_OP_N, tcg.TCG_OP_N, m, n, k, 1.0, At.cuda(), f.code, m,
                              Bt.cuda(), f.code, k, 0.0, D, tcg.TCG_R_32F, m, f.compute))
    got = D.cpu().numpy().T                                          # (m, n)
    want = oracle.dot_model(_raw(At, kind), ORACLE_TYPE[kind], _raw(Bt, kind),
                            ORACLE_TYPE[kind], m, n, k, tf32=(kind == "tf32"), **params)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    bad = np.argwhere(~same)
    assert bad.size == 0, (f"{len(bad)} of {m * n} differ; first (i, j, gpu, model): " +
                           str([(int(i), int(j), float(got[i, j]), float(want[i, j]))
                                for i, j in bad[:5]]))


@pytest.mark.timeout(900)
@pytest.mark.parametrize("kind", ["f16", "bf16"])
def test_issm_large_uniform_sample(features, kind):
    # ~6.6e4 dot products of length 1024 (the page's uniform sampling, section 3.2)
    params = features[kind].model_parameters()
    f = numerics.FORMATS[kind]
    m = n = 256
    k = 1024
    rng = np.random.default_rng(77 + KINDS.index(kind))
    At = _cast(rng.uniform(-1, 1, (k, m)), kind)
    Bt = _cast(rng.uniform(-1, 1, (n, k)), kind)
    D = torch.zeros((n, m), dtype=torch.float32, device="cuda:0")
    h = tcg.Handle()
    tcg.check(tcg.tcg_set_split_k(h.h, 1))        # one accumulation per output, no K split
    tcg.check(tcg.tcg_gemm_ex(h.h, tcg.TCG_OP_N, tcg.TCG_OP_N, m, n, k, 1.0, At.cuda(), f.code, m,
                              Bt.cuda(), f.code, k, 0.0, D, tcg.TCG_R_32F, m, f.compute))
    got = D.cpu().numpy().T
    want = oracle.dot_model(_raw(At, kind), ORACLE_TYPE[kind], _raw(Bt, kind),
                            ORACLE_TYPE[kind], m, n, k, **params)
    assert np.array_equal(got, want)


# --- ISSM at the page's scale -----------------------------------------------------------
#
# Section 3.2 of the page samples each format with 10^5 normal and 10^7 uniform inputs,
# plus directed special values (Inf, NaN, zeros, subnormals).  Here every output element is
# one dot product at the instruction's K (16 FP16/BF16, 8 TF32, 32 FP8): one strided-batched
# GEMM of `batch` independent 256 x 256 problems gives batch x 65536 dot products, built
# from batch x 512 independently drawn row and column vectors.  Every GPU result must equal
# the block-FMA model's (oracle.MODEL) bit for bit, by value class.

def _issm_batched(kind, A64, B64, batch, m, n):
    """GPU and model results for `batch` column-major problems A_b (m x k), B_b (k x n) given
    as float64 arrays of shape (batch, k, m) (A_b^T row-major) and (batch, n, k)."""
    f = numerics.FORMATS[kind]
    k = f.k_instr
    At = _cast(A64.reshape(batch * k, m), kind)
    Bt = _cast(B64.reshape(batch * n, k), kind)
    D = torch.zeros((batch, n, m), dtype=torch.float32, device="cuda:0")
    h = tcg.Handle()
    tcg.check(tcg.tcg_set_split_k(h.h, 1))        # one accumulation per output, no K split
    tcg.check(tcg.tcg_gemm_strided_batched(
        h.h, tcg.TCG_OP_N, tcg.TCG_OP_N, m, n, k, 1.0, At.cuda(), f.code, m, m * k,
        Bt.cuda(), f.code, k, k * n, 0.0, D, tcg.TCG_R_32F, m, m * n, batch, f.compute))
    tcg.check(tcg.tcg_get_device_error(h.h))
    got = D.cpu().numpy()
    h.close()
    Araw, Braw = _raw(At, kind).reshape(-1), _raw(Bt, kind).reshape(-1)
    per_a, per_b = m * k, k * n
    bad = 0
    first = []
    for b in range(batch):
        want = oracle.dot_model(Araw[b * per_a:(b + 1) * per_a], ORACLE_TYPE[kind],
                                Braw[b * per_b:(b + 1) * per_b], ORACLE_TYPE[kind], m, n, k,
                                tf32=(kind == "tf32"), **oracle.MODEL[ORACLE_TYPE[kind]])
        g = got[b].T
        same = (g == want) | (np.isnan(g) & np.isnan(want))
        if not same.all():
            idx = np.argwhere(~same)
            bad += len(idx)
            first += [(b, int(i), int(j), float(g[i, j]), float(want[i, j])) for i, j in idx[:2]]
    return bad, first[:6]


def _specials(kind):
    """Directed values of a format: infinities (where it has them), NaN, signed zeros,
    the smallest and largest subnormal, the smallest normal, and magnitudes whose
    products stay inside FP32."""
    f = numerics.FORMATS[kind]
    sub_min = 2.0 ** (f.emin - f.mbits)
    sub_max = (2.0 ** f.mbits - 1) * sub_min
    vals = [np.nan, 0.0, -0.0, sub_min, -sub_min, sub_max, 2.0 ** f.emin, -2.0 ** f.emin]
    if kind != "e4m3":                            # E4M3 (fn) has no infinities
        vals += [np.inf, -np.inf]
    big = min(f.emax, 60)
    vals += [2.0 ** big, -(2.0 ** big) * (1 + 2.0 ** -f.mbits)]
    return np.array(vals)


ISSM_M = ISSM_N = 256


@pytest.mark.timeout(900)
@pytest.mark.parametrize("kind", KINDS)
def test_issm_page_scale(features, kind):
    f = numerics.FORMATS[kind]
    k, m, n = f.k_instr, ISSM_M, ISSM_N
    rng = np.random.default_rng(9000 + KINDS.index(kind))
    counts = {}
    # 10^5 normal inputs: 2 problems of 256 x 256 dot products
    # 10^7 uniform inputs: 160 problems (1.05e7 dot products)
    # directed special values: 8 problems, each input a special value with probability 1/8
    for dist, batch in (("normal", 2), ("uniform", 160), ("directed", 8)):
        if dist == "directed":
            sp = _specials(kind)
            A = rng.uniform(-1, 1, (batch, k, m))
            B = rng.uniform(-1, 1, (batch, n, k))
            for X in (A, B):
                pick = rng.random(X.shape) < 0.125
                X[pick] = sp[rng.integers(0, len(sp), int(pick.sum()))]
        else:
            A = _draw(kind, dist, (batch, k, m), rng)
            B = _draw(kind, dist, (batch, n, k), rng)
        bad, first = _issm_batched(kind, A, B, batch, m, n)
        assert bad == 0, (f"{kind} {dist}: {bad} of {batch * m * n} differ from the model; "
                          f"first (batch, i, j, gpu, model): {first}")
        counts[dist] = batch * m * n
    print(f"ISSM {kind}: dot products of length {k} checked bit for bit: {counts}")
    assert counts["normal"] >= 10 ** 5 and counts["uniform"] >= 10 ** 7
