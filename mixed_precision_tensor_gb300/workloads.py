"""Seeded synthetic inputs for the GEMM workloads.

This module only draws numbers: it holds none of the GEMM's arithmetic and is
shared by the tests, the smoke check and the benchmark, so that the CUDA path
and the CPU oracle see the same bits.  Every matrix is drawn on the host with
``numpy.random.default_rng(seed)`` in the order A, then B, then C, row-major
(A is m x k, B is k x n, C is m x n), and converted to its storage type with
numpy (FP16) or torch (BF16) round-to-nearest-even casts.

Storage conventions of the returned arrays:
  * FP16 -> numpy float16
  * BF16 -> numpy uint16 holding the bfloat16 bit pattern
  * FP8 (E4M3 / E5M2) -> numpy uint8 holding the bit pattern (torch casts)
  * FP32 -> numpy float32
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    m: int
    n: int
    k: int
    in_type: str        # "f16" | "bf16" | "e4m3" | "e5m2" | "f32" (f32 means TF32 compute)
    out_type: str       # "f32" | "f16" | "bf16"
    alpha: float
    beta: float
    batch: int
    seed: int
    dist: str           # input distribution recipe, see draw()
    compute: str = ""   # "" (the input type's default) or "3xtf32" (FP32 as two TF32 words)

    @property
    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.k * self.batch

    def algorithmic_bytes(self) -> int:
        """A and B read once, C read once when beta != 0, D written once."""
        ein = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}[self.in_type]
        eout = {"f16": 2, "bf16": 2, "f32": 4}[self.out_type]
        per = (self.m * self.k + self.k * self.n) * ein + self.m * self.n * eout
        if self.beta != 0.0:
            per += self.m * self.n * eout
        return per * self.batch


# The five synthetic workloads.  Names state what they are.
WORKLOADS = {
    "fp16_gemm_256": Workload("fp16_gemm_256", 256, 256, 256, "f16", "f32", 1.0, 1.0, 1, 0,
                              "uniform"),
    "fp16_gemm_8192": Workload("fp16_gemm_8192", 8192, 8192, 8192, "f16", "f32", 1.0, 0.0, 1,
                               1, "uniform"),
    "bf16_proj_16384x4096x4096": Workload("bf16_proj_16384x4096x4096", 16384, 4096, 4096,
                                          "bf16", "f32", 1.0, 1.0, 1, 2, "proj"),
    "tf32_gemm_4096x4096x16384": Workload("tf32_gemm_4096x4096x16384", 4096, 4096, 16384,
                                          "f32", "f32", 1.0, 0.0, 1, 3, "uniform"),
    "fp16_batched_512x256": Workload("fp16_batched_512x256", 256, 256, 256, "f16", "f16", 1.0,
                                     0.5, 512, 4, "pow2"),
    # not one of the five above: FP8 inputs on the headline shape, the multi-word (3xTF32)
    # variant of the TF32 workload, and a split-K shape
    "fp8e4m3_gemm_8192": Workload("fp8e4m3_gemm_8192", 8192, 8192, 8192, "e4m3", "f32", 1.0,
                                  0.0, 1, 1, "uniform"),
    "fp32_3xtf32_4096x4096x16384": Workload("fp32_3xtf32_4096x4096x16384", 4096, 4096, 16384,
                                            "f32", "f32", 1.0, 0.0, 1, 3, "uniform",
                                            "3xtf32"),
    # one 256 x 256 output tile with a long K: the split-K case
    "fp16_splitk_256x256x65536": Workload("fp16_splitk_256x256x65536", 256, 256, 65536, "f16",
                                          "f32", 1.0, 0.0, 1, 5, "uniform"),
}
# Canonical order: small check case first, the headline case second.
WORKLOAD_ORDER = list(WORKLOADS)[:5]
HEADLINE = "fp16_gemm_8192"


def custom(m, n, k, in_type="f16", out_type="f32", alpha=1.0, beta=0.0, batch=1, seed=0,
           dist="uniform") -> Workload:
    return Workload(f"custom_{m}x{n}x{k}_{in_type}_{out_type}_b{batch}", m, n, k, in_type,
                    out_type, float(alpha), float(beta), batch, seed, dist)


def with_dist(w: Workload, dist: str) -> Workload:
    return replace(w, dist=dist, name=w.name + "_" + dist)


def _to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _to_fp8_bits(x32: np.ndarray, t: str) -> np.ndarray:
    import torch
    dt = torch.float8_e4m3fn if t == "e4m3" else torch.float8_e5m2
    tt = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return tt.to(dt).view(torch.uint8).numpy()


def _to_storage(x: np.ndarray, t: str) -> np.ndarray:
    if t in ("e4m3", "e5m2"):
        return _to_fp8_bits(x.astype(np.float32), t)
    if t == "f16":
        return x.astype(np.float32).astype(np.float16)
    if t == "bf16":
        return _to_bf16_bits(x.astype(np.float32))
    return x.astype(np.float32)


def _pow2_values(rng, shape):
    """sign * 2^e * (1 + mant/1024): e uniform integer in [-14, 4], mant uniform
    integer in [0, 1023], sign +-1 with equal odds -- exact FP16 normals."""
    e = rng.integers(-14, 5, size=shape)
    mant = rng.integers(0, 1024, size=shape)
    s = rng.integers(0, 2, size=shape) * 2 - 1
    return s * np.ldexp(1.0 + mant / 1024.0, e)


def draw(w: Workload):
    """Draw (A, B, C) for workload ``w``: shapes (batch, m, k), (batch, k, n),
    (batch, m, n); C is None when beta == 0 (it is never read then).

    Distributions (``w.dist``):
      uniform  A, B ~ U[-1, 1]; C ~ N(0, 1)
      proj     A ~ N(0, 1); B ~ N(0, 0.02) (standard deviation); C ~ N(0, 1)
      pow2     A, B as in _pow2_values; C ~ N(0, 1)
      integer  A, B uniform integers in {-2..2}; C ~ N(0, 1) for FP32 output
               with beta == 1 and k <= 256, else integer-valued C in {-8..8}
               (half-integers in {-8, -7.5, ..., 8} for FP16/BF16 output)
    C is drawn in FP64 and rounded to the output storage type.
    """
    rng = np.random.default_rng(w.seed)
    sa, sb, sc = (w.batch, w.m, w.k), (w.batch, w.k, w.n), (w.batch, w.m, w.n)
    if w.dist == "uniform":
        A = rng.uniform(-1.0, 1.0, sa)
        B = rng.uniform(-1.0, 1.0, sb)
    elif w.dist == "proj":
        A = rng.standard_normal(sa)
        B = rng.normal(0.0, 0.02, sb)
    elif w.dist == "pow2":
        A = _pow2_values(rng, sa)
        B = _pow2_values(rng, sb)
    elif w.dist == "integer":
        A = rng.integers(-2, 3, sa).astype(np.float64)
        B = rng.integers(-2, 3, sb).astype(np.float64)
    else:
        raise ValueError(w.dist)
    A = _to_storage(A, w.in_type)
    B = _to_storage(B, w.in_type)
    C = None
    if w.beta != 0.0:
        if w.dist == "integer" and not (w.out_type == "f32" and w.beta == 1.0 and w.k <= 256):
            if w.out_type == "f32":
                C = rng.integers(-8, 9, sc).astype(np.float64)
            else:
                C = rng.integers(-16, 17, sc) / 2.0
        else:
            C = rng.standard_normal(sc)
        C = _to_storage(C, w.out_type)
    return A, B, C


def sample_tiles(m, n, count=64, tile=128, seed=0):
    """Seeded choice of ``count`` output tiles (tile x tile, the last row/column
    of tiles may be ragged) of an m x n result, always including the four
    corner tiles.  Returns a list of (i0, i1, j0, j1) in row-major terms."""
    tm, tn = -(-m // tile), -(-n // tile)
    corners = {(0, 0), (0, tn - 1), (tm - 1, 0), (tm - 1, tn - 1)}
    rng = np.random.default_rng(seed + 10000)
    picks = list(dict.fromkeys(sorted(corners)))
    total = tm * tn
    want = min(count, total)
    while len(picks) < want:
        t = int(rng.integers(0, total))
        cand = (t // tn, t % tn)
        if cand not in picks:
            picks.append(cand)
    return [(a * tile, min((a + 1) * tile, m), b * tile, min((b + 1) * tile, n))
            for a, b in picks]
