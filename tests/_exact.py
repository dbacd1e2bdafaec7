"""Independent exact helpers for pinning the oracle.

Nothing here shares code with ``oracle/``: decoding goes through torch's own
float8 dtypes, sums are exact rationals (``fractions.Fraction``) or float64
sums proven exact, and rounding to BF16 is a search over the explicit grid of
all finite BF16 numbers (every BF16 value and every midpoint between two
neighbours is exactly representable in float64 and as a Fraction).
"""
from __future__ import annotations

import bisect
from fractions import Fraction
from functools import lru_cache

import numpy as np
import torch

BF16_INF = 0x7F80
BF16_MAX = 0x7F7F


def e4m3_values(codes) -> np.ndarray:
    """float64 values of E4M3 code bytes via torch.float8_e4m3fn (exact)."""
    t = torch.as_tensor(np.ascontiguousarray(np.asarray(codes, dtype=np.uint8)))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e5m2_values(codes) -> np.ndarray:
    """float64 values of E5M2 code bytes via torch.float8_e5m2 (exact; +-inf and NaN kept)."""
    t = torch.as_tensor(np.ascontiguousarray(np.asarray(codes, dtype=np.uint8)))
    return t.view(torch.float8_e5m2).to(torch.float64).numpy()


def values_of(codes, fmt: str) -> np.ndarray:
    return e5m2_values(codes) if fmt == "e5m2" else e4m3_values(codes)


def e8m0_values(codes) -> np.ndarray:
    """float64 values 2^(c-127) of E8M0 bytes via torch.float8_e8m0fnu (exact)."""
    t = torch.as_tensor(np.ascontiguousarray(np.asarray(codes, dtype=np.uint8)))
    return t.view(torch.float8_e8m0fnu).to(torch.float64).numpy()


@lru_cache(maxsize=1)
def _grid():
    bits = np.arange(0, BF16_INF, dtype=np.uint32)          # +0 .. max finite
    vals = (bits << 16).view(np.float32).astype(np.float64)
    return bits.astype(np.uint16), vals


@lru_cache(maxsize=1)
def _grid_fractions():
    _, vals = _grid()
    return [Fraction(float(v)) for v in vals]


def _pick(lo_bits: int, hi_bits: int, below: bool, above: bool) -> int:
    if below:
        return lo_bits
    if above:
        return hi_bits
    return lo_bits if lo_bits % 2 == 0 else hi_bits       # tie: even significand


def round_fraction_to_bf16(x: Fraction) -> int:
    """BF16 bits nearest to the exact rational x (ties to even, overflow to inf)."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    fr = _grid_fractions()
    i = bisect.bisect_right(fr, a) - 1                     # fr[i] <= a
    if fr[i] == a:
        return sign | i
    lo = fr[i]
    hi = fr[i + 1] if i + 1 < len(fr) else Fraction(2) ** 128
    mid = (lo + hi) / 2
    return sign | _pick(i, i + 1, a < mid, a > mid)


def round_f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Vectorised exact rounding of float64 values (taken as exact) to BF16 bits."""
    bits, vals = _grid()
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    i = np.searchsorted(vals, a, side="right") - 1
    lo = vals[i]
    top = 2.0 ** 128
    hi = np.where(i + 1 < len(vals), vals[np.minimum(i + 1, len(vals) - 1)], top)
    mid = (lo + hi) / 2                                    # exact: <= 9 significant bits
    lo_b = i.astype(np.int64)
    hi_b = lo_b + 1                                        # BF16_INF when i is the max
    tie_even = np.where(lo_b % 2 == 0, lo_b, hi_b)
    out = np.where(a == lo, lo_b, np.where(a < mid, lo_b, np.where(a > mid, hi_b, tie_even)))
    out = np.where(x < 0, out | 0x8000, out)             # negative underflow gives -0
    return out.astype(np.uint16)


def exact_gemm_fraction(A_seg, A_sf, B, B_sf, a_fmt: str = "e4m3", b_fmt: str = "e4m3") -> np.ndarray:
    """Brute-force exact C (BF16 bits) with rational arithmetic; tiny shapes, finite codes only."""
    R = len(A_seg)
    M, ka = np.asarray(A_seg[0]).shape
    N, K = np.asarray(B).shape
    av = np.concatenate([values_of(a, a_fmt) for a in A_seg], axis=1)     # [M][K]
    asf = np.concatenate([np.asarray(s, dtype=np.uint8) for s in A_sf], axis=1)
    bv = values_of(B, b_fmt)
    bsf = np.asarray(B_sf, dtype=np.uint8)
    out = np.zeros((M, N), dtype=np.uint16)
    two = Fraction(2)
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                if av[m, k] == 0 or bv[n, k] == 0:
                    continue
                ea = int(asf[m, k // 32]) - 127
                eb = int(bsf[n, k // 32]) - 127
                s += Fraction(float(av[m, k])) * Fraction(float(bv[n, k])) * two ** (ea + eb)
            out[m, n] = round_fraction_to_bf16(s)
    return out
