"""Pins of the oracle's number-format routines (CPU only).

Each routine is checked against something other than itself: numpy/torch
conversions (library routines), closed-form tie cases, and for TF32 an
exhaustive comparison over all 2^32 FP32 patterns with a second formulation in
integer bit arithmetic (tests/native/tf32_bits_check.c).
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f64(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


@pytest.mark.parametrize("name,fn,tdt", [("e4m3", "f8e4m3_to_f64", "float8_e4m3fn"),
                                         ("e5m2", "f8e5m2_to_f64", "float8_e5m2")])
def test_f8_decode_all_patterns_match_torch(name, fn, tdt):
    bits = np.arange(256, dtype=np.uint8)
    got = getattr(oracle, fn)(bits)
    want = torch.from_numpy(bits).view(getattr(torch, tdt)).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_f8_closed_forms():
    e4 = oracle.f8e4m3_to_f64(np.array([0x7E, 0x01, 0x08, 0x38, 0xFE, 0x7F], dtype=np.uint8))
    assert e4[0] == 448.0 and e4[1] == 2.0 ** -9 and e4[2] == 2.0 ** -6 and e4[3] == 1.0
    assert e4[4] == -448.0 and np.isnan(e4[5])
    e5 = oracle.f8e5m2_to_f64(np.array([0x7B, 0x01, 0x3C, 0x7C, 0x7D], dtype=np.uint8))
    assert e5[0] == 57344.0 and e5[1] == 2.0 ** -16 and e5[2] == 1.0
    assert e5[3] == np.inf and np.isnan(e5[4])


def _f16_edge_values():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    v = h.astype(np.float64)
    v = v[np.isfinite(v)]
    v = np.unique(v)
    mids = (v[:-1] + v[1:]) / 2.0                       # exact ties in FP64
    near = np.concatenate([np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf)])
    extra = np.array([65504.0, 65519.999, 65520.0, 65536.0, 1e6, 2.0 ** -25, 3 * 2.0 ** -25,
                      2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 0.0, -0.0, np.inf,
                      -np.inf, 1e-300])
    return np.concatenate([v, mids, near, extra, -extra])


def test_f64_to_f16_rne_matches_numpy():
    rng = np.random.default_rng(7)
    rand = np.concatenate([
        rng.standard_normal(3_000_000) * 100.0,
        np.ldexp(rng.uniform(1, 2, 3_000_000), rng.integers(-30, 18, 3_000_000)),
        rng.uniform(-1e-4, 1e-4, 2_000_000),
    ])
    x = np.concatenate([_f16_edge_values(), rand])
    got = oracle.f64_to_f16_bits(x)
    want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_f16_rne_nan_and_ties_closed_form():
    got = oracle.f64_to_f16_bits([np.nan, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0])
    assert got[0] & 0x7C00 == 0x7C00 and got[0] & 0x3FF != 0
    # ties go to the even neighbour
    assert got[1] == 0x3C00                 # 1 + 2^-11 -> 1
    assert got[2] == 0x3C02                 # 1 + 3*2^-11 -> 1 + 2^-9
    assert got[3] == np.float16(2048).view(np.uint16)
    assert got[4] == np.float16(2052).view(np.uint16)


def test_f64_to_bf16_rne_matches_torch_on_float32_values():
    # Values exactly representable in FP32 so torch's float32 -> bfloat16 cast is
    # a single rounding of the same value.
    rng = np.random.default_rng(8)
    f32 = np.concatenate([
        rng.standard_normal(2_000_000).astype(np.float32),
        np.ldexp(rng.uniform(1, 2, 1_000_000), rng.integers(-140, 128, 1_000_000)).astype(np.float32),
        rng.integers(0, 1 << 32, 2_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    f32 = f32[~np.isnan(f32)]
    # exact ties: bf16 value + half a bf16 ulp
    base = rng.integers(0, 1 << 15, 100_000).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    x = np.concatenate([f32, ties])
    got = oracle.f64_to_bf16_bits(x.astype(np.float64))
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_overflow_and_subnormals():
    mx = (2.0 - 2.0 ** -7) * 2.0 ** 127
    half_ulp = 2.0 ** (127 - 8)
    got = oracle.f64_to_bf16_bits([mx, mx + half_ulp, mx + half_ulp * 0.99, 2.0 ** -133,
                                   2.0 ** -134, 3 * 2.0 ** -134])
    assert got[0] == 0x7F7F
    assert got[1] == 0x7F80                 # tie with odd max -> Inf
    assert got[2] == 0x7F7F
    assert got[3] == 0x0001                 # smallest subnormal
    assert got[4] == 0x0000                 # tie -> even (zero)
    assert got[5] == 0x0002                 # tie -> even (2)


def test_f64_to_f32_matches_numpy():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(1_000_000) * 1e3,
                        np.ldexp(rng.uniform(1, 2, 500_000), rng.integers(-160, 130, 500_000))])
    got = oracle.f64_to_f32(x)
    want = x.astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_tf32_closed_form_ties():
    one = np.float32(1.0).view(np.uint32)
    cases = {
        int(one) + (1 << 12): 0x3F800000,    # 1 + 2^-11: tie -> even -> 1
        int(one) + (3 << 12): 0x3F804000,    # 1 + 3*2^-11: tie -> even -> 1 + 2^-9
        int(one) + (1 << 12) + 1: 0x3F802000,  # just past the tie -> up
        0x7F7FFFFF: 0x7F800000,              # max finite FP32 -> past TF32 max -> Inf
        0x7F800000: 0x7F800000,              # +Inf
        0xFF800000: 0xFF800000,              # -Inf
        0x00001000: 0x00000000,              # subnormal tie -> even (0)
        0x00003000: 0x00004000,              # subnormal tie -> even
        0x80000000: 0x80000000,              # -0
    }
    got = oracle.tf32_round_bits(np.array(list(cases), dtype=np.uint32))
    assert [int(g) for g in got] == list(cases.values())
    nan = oracle.tf32_round_bits(np.array([0x7F800001, 0xFFC00001], dtype=np.uint32))
    for v in nan:
        assert (v & 0x7F800000) == 0x7F800000 and (v & 0x007FE000) != 0


def _build_checker():
    out = os.path.join(HERE, "native", "_build")
    os.makedirs(out, exist_ok=True)
    src = os.path.join(HERE, "native", "tf32_bits_check.c")
    lib = os.path.join(out, "libtf32check.so")
    if not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        tmp = lib + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, src], check=True)
        os.replace(tmp, lib)
    return ctypes.CDLL(lib)


@pytest.mark.timeout(600)
def test_tf32_rounding_exhaustive_against_bit_formulation():
    chk = _build_checker()
    chk.tf32_exhaustive_mismatches.restype = ctypes.c_uint64
    chk.tf32_exhaustive_mismatches.argtypes = [ctypes.c_void_p, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_uint32)]
    first = ctypes.c_uint32(0)
    bad = chk.tf32_exhaustive_mismatches(ctypes.c_void_p(oracle.tf32_round_fn_address()),
                                         os.cpu_count() or 1, ctypes.byref(first))
    assert bad == 0, f"{bad} mismatches, first at 0x{first.value:08x}"
