"""Test-side helpers: golden-file parsing, the row-major -> column-major call
mapping, and the element-wise acceptance bound.  Test code only."""
from __future__ import annotations

import os
import re
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

TYPE_CODE = {"f16": oracle.F16, "bf16": oracle.BF16, "f32": oracle.F32,
             "e4m3": oracle.F8E4M3, "e5m2": oracle.F8E5M2}


def raw(x: np.ndarray) -> np.ndarray:
    """Raw storage view: FP16 as uint16 bits, BF16 already uint16, FP32 as is."""
    if x.dtype == np.float16:
        return x.view(np.uint16)
    return x


def parse_term(t: str) -> Fraction:
    total = Fraction(0)
    for part in t.split("+"):
        part = part.strip()
        mo = re.fullmatch(r"(-?\d+)\*2\^(-?\d+)", part)
        if mo:
            total += Fraction(int(mo.group(1))) * Fraction(2) ** int(mo.group(2))
        else:
            total += Fraction(part)
    return total


def load_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals = [parse_term(v) for v in val.split(",")]
            out[key] = vals if len(vals) > 1 or key in ("a", "b") else vals[0]
    return out


def oracle_rowmajor(w, A, B, C, b=0, rows=None, cols=None, nthreads=None):
    """Oracle for the row-major problem D = alpha*A@B + beta*C of workload ``w``
    (batch entry ``b``), through the column-major call that the library gets:
    gemm(N, N, n, m, k, alpha, B, ldb=n, A, lda=k, beta, C, ldc=n).
    ``rows``/``cols`` select a block of the row-major D.  Returns (D, R, absAB)
    as row-major blocks."""
    m, n, k = w.m, w.n, w.k
    i0, i1 = rows if rows else (0, m)
    j0, j1 = cols if cols else (0, n)
    Ab = raw(A[b]).reshape(-1)
    Bb = raw(B[b]).reshape(-1)
    Cb = raw(C[b]).reshape(-1) if C is not None else None
    D, R, AB = oracle.gemm(oracle.OP_N, oracle.OP_N, n, m, k, w.alpha, Bb,
                           TYPE_CODE[w.in_type], n, Ab, TYPE_CODE[w.in_type], k, w.beta, Cb,
                           TYPE_CODE[w.out_type], n, tf32=(w.in_type == "f32"),
                           rows=(j0, j1), cols=(i0, i1), nthreads=nthreads)
    return D.T, R.T, AB.T


def model_block(args, rows, cols, plan=None, batch_entry=0, tf32=False, nthreads=None,
                **params):
    """oracle.gemm_model over the block rows x cols of a column-major call (``args`` =
    transa, transb, m, n, k, alpha, A, atype, lda, B, btype, ldb, beta, C, ctype, ldc),
    each output tile with the K ranges the library gave it: ``plan`` = (tile_m, tile_n,
    splits, k_per_split) from tcg_gemm_tile_plan (None: one accumulation over all of K)."""
    i0, i1 = rows
    j0, j1 = cols
    if plan is None:
        return oracle.gemm_model(*args, tf32=tf32, rows=rows, cols=cols, nthreads=nthreads,
                                 **params)
    tm, tn, splits, kps = plan
    out = None
    for ti in range(i0 // tm, (i1 - 1) // tm + 1):
        for tj in range(j0 // tn, (j1 - 1) // tn + 1):
            r0, r1 = max(i0, ti * tm), min(i1, (ti + 1) * tm)
            c0, c1 = max(j0, tj * tn), min(j1, (tj + 1) * tn)
            s = int(splits[batch_entry, ti, tj])
            D = oracle.gemm_model(*args, tf32=tf32, rows=(r0, r1), cols=(c0, c1),
                                  nthreads=nthreads, splits=s,
                                  k_per_split=int(kps[batch_entry, ti, tj]) if s > 1 else 0,
                                  **params)
            if out is None:
                out = np.zeros((i1 - i0, j1 - j0), dtype=D.dtype)
            out[r0 - i0:r1 - i0, c0 - j0:c1 - j0] = D
    return out


def model_rowmajor(w, A, B, C, b=0, rows=None, cols=None, nthreads=None, plan=None):
    """The block-FMA model (oracle.MODEL parameters) for the same row-major problem
    and block as :func:`oracle_rowmajor`, with the library's per-tile K ranges ``plan``
    (tcg_gemm_tile_plan of the column-major call, or None).  Returns D as a row-major
    block."""
    m, n, k = w.m, w.n, w.k
    i0, i1 = rows if rows else (0, m)
    j0, j1 = cols if cols else (0, n)
    Ab = raw(A[b]).reshape(-1)
    Bb = raw(B[b]).reshape(-1)
    Cb = raw(C[b]).reshape(-1) if C is not None else None
    t = TYPE_CODE[w.in_type]
    args = (oracle.OP_N, oracle.OP_N, n, m, k, w.alpha, Bb, t, n, Ab, t, k, w.beta, Cb,
            TYPE_CODE[w.out_type], n)
    D = model_block(args, (j0, j1), (i0, i1), plan=plan, batch_entry=b,
                    tf32=(w.in_type == "f32"), nthreads=nthreads, **oracle.MODEL[t])
    return D.T


def decode_out(x: np.ndarray, out_type: str) -> np.ndarray:
    if out_type == "f16":
        return x.view(np.float16).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)
    if out_type == "bf16":
        return oracle.bf16_to_f64(x.view(np.uint16))
    return x.astype(np.float64)


def ulp16(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14)
    u = np.ldexp(1.0, (e - 10).astype(np.int64))
    return np.where(a > 0, u, 2.0 ** -24)


def ulpbf16(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    u = np.ldexp(1.0, (e - 7).astype(np.int64))
    return np.where(a > 0, u, 2.0 ** -133)


def check_bound(got, ref, absab, cval, k, alpha, beta, out_type):
    """Element-wise acceptance: |D - ref| <= k*2^-23*(|alpha|*(|A||B|) + |beta|*|C|)
    plus one output ulp for 16-bit outputs; NaN == NaN, Inf signs must match.
    ``got``/``ref`` are decoded FP64 arrays, ``cval`` the decoded C (or None).
    Returns (ok, worst normalised error, index of worst)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    cterm = np.abs(beta) * np.abs(cval) if (cval is not None and beta != 0) else 0.0
    bound = k * 2.0 ** -23 * (abs(alpha) * absab + cterm)
    if out_type == "f16":
        bound = bound + ulp16(ref)
    elif out_type == "bf16":
        bound = bound + ulpbf16(ref)
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    if not np.array_equal(nan_ref, nan_got):
        return False, np.inf, int(np.argmax(nan_ref != nan_got))
    inf_ref = np.isinf(ref)
    if not np.array_equal(inf_ref, np.isinf(got)) or not np.array_equal(
            np.sign(ref[inf_ref]), np.sign(got[inf_ref])):
        return False, np.inf, int(np.argmax(inf_ref != np.isinf(got)))
    fin = ~(nan_ref | inf_ref)
    err = np.zeros_like(ref)
    err[fin] = np.abs(got[fin] - ref[fin])
    with np.errstate(divide="ignore", invalid="ignore"):
        norm = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                        np.where(err > 0, np.inf, 0.0))
    worst = float(norm.max()) if norm.size else 0.0
    return bool(worst <= 1.0), worst, int(np.argmax(norm)) if norm.size else 0


def values_equal(got, ref):
    """Bit-exactness by value class: NaN == NaN, +0 == -0, otherwise equal."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_nan = np.isnan(got) & np.isnan(ref)
    return bool(np.all(both_nan | (got == ref)))
