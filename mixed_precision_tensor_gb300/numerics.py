"""Numeric-feature probe of the tensor core, run through the library's own GEMM.

"NVIDIA Tensor Core混合精度计算原理与应用解析", section 3.1 (GNFT): hand-built test vectors,
each aimed at one feature of the hardware's arithmetic, are run through the tensor core
and the outputs identify the feature: the block FMA size (section 2.2.2), the width of
the accumulator's alignment window (section 2.2.1), how intermediate and final sums are
rounded (section 2.3) and how subnormals are treated (section 2.2.3).

Every vector here is a dot product d = sum_p a_p b_p with alpha = 1, beta = 0 and an FP32
result, so d is the tensor core's accumulator itself.  Many vectors share one GEMM call:
test i is row i of A and column i of B, and its result is D[i, i].  All inputs are
exactly representable in the probed format, and every expected outcome is a closed form
of the vector (no model is evaluated here).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from . import (TCG_COMPUTE_32F, TCG_COMPUTE_32F_FAST_TF32, TCG_OP_N, TCG_R_16BF, TCG_R_16F,
               TCG_R_32F, TCG_R_8F_E4M3, TCG_R_8F_E5M2, Handle, check, tcg_gemm_ex)


@dataclass(frozen=True)
class Format:
    name: str
    dtype: torch.dtype
    code: int
    compute: int
    k_instr: int          # K of one tcgen05.mma instruction of this kind
    emin: int             # smallest normal exponent
    emax: int             # largest normal exponent
    mbits: int            # stored mantissa bits
    base: int             # exponent of the "unit" the vectors are built around
    jmax: int             # smallest term used: unit * 2^-jmax


FORMATS = {
    "f16": Format("f16", torch.float16, TCG_R_16F, TCG_COMPUTE_32F, 16, -14, 15, 10, 8, 36),
    "bf16": Format("bf16", torch.bfloat16, TCG_R_16BF, TCG_COMPUTE_32F, 16, -126, 127, 7, 0, 60),
    "tf32": Format("tf32", torch.float32, TCG_R_32F, TCG_COMPUTE_32F_FAST_TF32, 8, -126, 127, 10,
                   0, 60),
    "e4m3": Format("e4m3", torch.float8_e4m3fn, TCG_R_8F_E4M3, TCG_COMPUTE_32F, 32, -6, 8, 3, 16,
                   28),
    "e5m2": Format("e5m2", torch.float8_e5m2, TCG_R_8F_E5M2, TCG_COMPUTE_32F, 32, -14, 15, 2, 16,
                   44),
}


@dataclass
class Features:
    """What the probe found for one input format (None: not determined)."""
    kind: str
    k_per_instruction: int
    block: int | None = None              # products aligned together (N_FMA)
    frac_bits: int | None = None          # cut: 2^-frac below the largest alignment exponent
    exponent: str | None = None           # "input-sum" or "product"
    accumulator_aligned: bool | None = None
    normalisation: str | None = None      # "toward-zero", "nearest-even", "down", "up"
    cut: str | None = None                # "toward-zero" or "floor"
    subnormal_inputs: bool | None = None
    subnormal_outputs: bool | None = None
    specials_ieee: bool | None = None
    notes: list = field(default_factory=list)

    def model_parameters(self):
        """Parameters of the block-FMA model these features describe, or None when a
        feature is missing or outside that model (floor cut, unaligned accumulator,
        directed normalisation)."""
        if None in (self.block, self.frac_bits, self.exponent, self.accumulator_aligned,
                    self.normalisation, self.cut):
            return None
        if self.cut != "toward-zero" or not self.accumulator_aligned:
            return None
        if self.normalisation not in ("toward-zero", "nearest-even"):
            return None
        return {"block": self.block, "frac": self.frac_bits,
                "norm_rne": self.normalisation == "nearest-even",
                "exp_sum": self.exponent == "input-sum"}


def _split(v: float, f: Format, m: float | None = None):
    """(a, b) with a * b == v, both normal numbers of format f.  v = s * mant * 2^e with
    mant in [1, 2) holding at most f.mbits fraction bits."""
    if v == 0.0:
        return 0.0, 0.0
    mant, e = math.frexp(abs(v))
    mant, e = mant * 2.0, e - 1
    e1 = e // 2
    e2 = e - e1
    while e1 < f.emin:
        e1, e2 = e1 + 1, e2 - 1
    while e2 < f.emin:
        e1, e2 = e1 - 1, e2 + 1
    while e1 > f.emax:
        e1, e2 = e1 - 1, e2 + 1
    while e2 > f.emax:
        e1, e2 = e1 + 1, e2 - 1
    if not (f.emin <= e1 <= f.emax and f.emin <= e2 <= f.emax):
        raise ValueError(f"{v} is not a product of two {f.name} normals")
    return math.copysign(mant * 2.0 ** e1, v), 2.0 ** e2


class _Runner:
    """Runs a batch of dot-product vectors through one GEMM call."""

    def __init__(self, handle: Handle, f: Format, device):
        self.h, self.f, self.dev = handle, f, device

    def run(self, tests, K):
        """tests: lists of terms, a term being a product value (split into two inputs)
        or an (a, b) pair; term p of test i goes to A[i, p] and B[p, i].  Returns the
        results as a list of floats."""
        f = self.f
        T = max(16, (len(tests) + 15) // 16 * 16)
        A = torch.zeros((K, T), dtype=torch.float64)     # column-major T x K
        B = torch.zeros((T, K), dtype=torch.float64)     # column-major K x T
        for i, terms in enumerate(tests):
            for p, t in enumerate(terms):
                a, b = t if isinstance(t, tuple) else _split(t, f)
                A[p, i] = a
                B[i, p] = b
        At = A.to(torch.float32).to(f.dtype)
        Bt = B.to(torch.float32).to(f.dtype)
        for x, ref in ((At, A), (Bt, B)):
            back = x.to(torch.float64)
            same = (back == ref) | (torch.isnan(back) & torch.isnan(ref))
            if not bool(same.all()):
                raise ValueError(f"probe input not exactly representable in {f.name}")
        At, Bt = At.to(self.dev), Bt.to(self.dev)
        D = torch.zeros((T, T), dtype=torch.float32, device=self.dev)
        check(tcg_gemm_ex(self.h.h, TCG_OP_N, TCG_OP_N, T, T, K, 1.0, At, f.code, T, Bt, f.code,
                          K, 0.0, D, TCG_R_32F, T, f.compute), "probe gemm")
        d = D.cpu().to(torch.float64)
        return [float(d[i, i]) for i in range(len(tests))]


def _step(flags):
    """Index of the first True in a list that is False...False True...True, else None."""
    if True not in flags:
        return len(flags)
    first = flags.index(True)
    return first if all(flags[first:]) and not any(flags[:first]) else None


def probe_format(handle: Handle, kind: str, device=None) -> Features:
    f = FORMATS[kind]
    dev = device or torch.device("cuda", torch.cuda.current_device())
    run = _Runner(handle, f, dev).run
    feat = Features(kind, f.k_instr)
    U = 2.0 ** f.base
    K = 4 * f.k_instr
    tiny = U * 2.0 ** -f.jmax

    # Block size: [U, -U, ..., tiny at p] -- tiny is cut inside the block of the pair and
    # survives once it is in a later block (the accumulator is then 0).
    ps = list(range(2, 2 * f.k_instr + 2))
    out = run([[U, -U] + [0.0] * (p - 2) + [tiny] for p in ps], K)
    bad = [o for o in out if o not in (0.0, tiny)]
    first = _step([o == tiny for o in out])
    if bad or first is None:
        feat.notes.append(f"block: no clean step ({out})")
    else:
        feat.block = ps[first] if first < len(ps) else None

    # Window: [U, -U, U 2^-j] -- U 2^-j survives while it is inside the window.
    js = list(range(1, f.jmax + 1))
    out = run([[U, -U, U * 2.0 ** -j] for j in js], K)
    kept = [o == U * 2.0 ** -j for o, j in zip(out, js)]
    bad = [o for o, j in zip(out, js) if o not in (0.0, U * 2.0 ** -j)]
    first = _step([not k for k in kept])
    if bad or first is None or first == 0:
        feat.notes.append(f"window: no clean step ({out})")
    elif first < len(js):
        feat.frac_bits = js[first - 1]
    else:
        feat.notes.append(f"window: wider than {f.jmax} bits")
    F = feat.frac_bits
    if F is None:
        return feat

    # Alignment exponent: 1.5 * 1.5 has input exponents summing to 0 but the product's
    # exponent is 1.  [P, -P, U 2^-F] keeps U 2^-F only with input-exponent sums.
    e1 = f.base // 2
    P = (1.5 * 2.0 ** e1, 1.5 * 2.0 ** (f.base - e1))
    NP = (-P[0], P[1])
    o = run([[P, NP, U * 2.0 ** -F]], K)[0]
    feat.exponent = ("input-sum" if o == U * 2.0 ** -F else "product" if o == 0.0 else None)
    if feat.exponent is None:
        feat.notes.append(f"exponent: unexpected {o}")

    # Accumulator: c = U from the first instruction; the next instruction adds
    # 2^(F-22) copies of U 2^-(F+1).  Aligned with c they are all cut (d = U); summed on
    # their own they make U 2^-23 and d = U (1 + 2^-23).
    ncopy = 2 ** (F - 22)
    if 1 <= ncopy <= f.k_instr:
        t = [U] + [0.0] * (f.k_instr - 1) + [U * 2.0 ** -(F + 1)] * ncopy
        control = [U] + [0.0] * (f.k_instr - 1) + [U * 2.0 ** -F] * (ncopy // 2 or 1)
        o, oc = run([t, control], K)
        want_c = U * (1 + 2.0 ** -F * (ncopy // 2 or 1))
        if oc != want_c:
            feat.notes.append(f"accumulator control: {oc} != {want_c}")
        elif o == U:
            feat.accumulator_aligned = True
        elif o == U * (1 + 2.0 ** -23):
            feat.accumulator_aligned = False
        else:
            feat.notes.append(f"accumulator: unexpected {o}")

    # Normalisation of the block sum: U (1 + 2^-23 + 2^-24) is 1.5 ulp above U.
    if F >= 24:
        t = [U, U * 2.0 ** -23, U * 2.0 ** -24]
        o, on = run([t, [-x for x in t]], K)
        lo, hi = U * (1 + 2.0 ** -23), U * (1 + 2.0 ** -22)
        table = {(lo, -lo): "toward-zero", (hi, -hi): "nearest-even", (lo, -hi): "down",
                 (hi, -lo): "up"}
        feat.normalisation = table.get((o, on))
        if feat.normalisation is None:
            feat.notes.append(f"normalisation: unexpected {o}, {on}")

    # Cut direction: [U, -U 2^-(F+1)]: toward zero drops the small term (d = U); a floor
    # cut turns it into -U 2^-F and d < U.
    o = run([[U, -U * 2.0 ** -(F + 1)]], K)[0]
    feat.cut = "toward-zero" if o == U else ("floor" if o < U else None)
    if feat.cut is None:
        feat.notes.append(f"cut: unexpected {o}")

    # Subnormal inputs: the smallest positive subnormal times a power of two.
    smallest = 2.0 ** (f.emin - f.mbits)
    scale = 2.0 ** min(f.emax, 20)
    o = run([[(smallest, scale)]], K)[0]
    feat.subnormal_inputs = (o == smallest * scale) if o in (0.0, smallest * scale) else None

    # Subnormal FP32 results (only reachable from BF16/TF32 products): 2^-70 * 2^-70.
    if f.emin <= -70:
        o = run([[(2.0 ** -70, 2.0 ** -70)]], K)[0]
        feat.subnormal_outputs = (o == 2.0 ** -140) if o in (0.0, 2.0 ** -140) else None

    # Special values, compared by class with IEEE arithmetic.
    nan = float("nan")
    tests, want = [[(nan, 1.0)]], ["nan"]
    if f.name != "e4m3":                  # E4M3 has no infinities
        inf = float("inf")
        tests += [[(inf, 1.0)], [(inf, 1.0), (-inf, 1.0)], [(inf, 0.0)]]
        want += ["+inf", "nan", "nan"]
    out = run(tests, K)
    cls = ["nan" if math.isnan(o) else ("+inf" if o == math.inf else
                                        "-inf" if o == -math.inf else "finite") for o in out]
    feat.specials_ieee = cls == want
    if not feat.specials_ieee:
        feat.notes.append(f"specials: {cls} != {want}")
    return feat


def probe(handle: Handle | None = None, kinds=tuple(FORMATS), device=None) -> dict:
    """Run the feature probe for every format in ``kinds`` on the current CUDA device.
    Returns {kind: Features}."""
    h = handle or Handle()
    return {k: probe_format(h, k, device) for k in kinds}
