"""Pins for the CPU oracle: each check ties it to something other than itself.

The operation (all_to_all_matmul_impl.h, MatmulProcess with split-K over the R
segments; all_to_all_comm_udma.h, PutSegmentToRank for where segment r lands)
is C = bf16(concat_r(A_r * sA_r) @ (B * sB)^T) with E4M3 operands and E8M0
scales per 32 along K.  The pins below are chosen so that a plausible mistake
in the oracle (a dropped term, a wrong sign, an index or segment offset off,
transposed operands, double rounding, a wrong scale bias) fails at least one.
"""
from __future__ import annotations

import json
import os
import random
import shutil
import subprocess
import ctypes
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from all_mxfp8_block_gb300 import inputs
from tests import _exact

HERE = os.path.dirname(os.path.abspath(__file__))


def _split(A_full, sf_full, R, ka):
    A = [np.ascontiguousarray(A_full[:, r * ka:(r + 1) * ka]) for r in range(R)]
    S = [np.ascontiguousarray(sf_full[:, r * ka // 32:(r + 1) * ka // 32]) for r in range(R)]
    return A, S


# --- decoders: exhaustive against torch's float8 dtypes ------------------------------

def test_e4m3_decode_exhaustive_vs_torch():
    ref = _exact.e4m3_values(np.arange(256))
    for c in range(256):
        got = oracle.decode_e4m3(c)
        if c in (0x7F, 0xFF):
            assert np.isnan(got) and np.isnan(ref[c])
        else:
            assert got == ref[c], (hex(c), got, ref[c])
    # closed-form landmarks of the "fn" flavour
    assert oracle.decode_e4m3(0x7E) == 448.0
    assert oracle.decode_e4m3(0x01) == 2.0 ** -9
    assert oracle.decode_e4m3(0x08) == 2.0 ** -6
    assert oracle.decode_e4m3(0x38) == 1.0


def test_e8m0_decode_exhaustive_vs_torch():
    ref = _exact.e8m0_values(np.arange(256))
    for c in range(256):
        got = oracle.decode_e8m0(c)
        if c == 0xFF:
            assert np.isnan(got) and np.isnan(ref[c])
        else:
            assert got == ref[c] == 2.0 ** (c - 127)


# --- the single rounding step, against a search over the BF16 grid --------------------

def test_e5m2_decode_exhaustive_vs_torch():
    """All 256 E5M2 codes against torch.float8_e5m2 (infinities and NaNs included)."""
    codes = np.arange(256, dtype=np.uint8)
    want = _exact.e5m2_values(codes)
    got = np.array([oracle.decode_e5m2(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[0x7C] == np.inf and got[0xFC] == -np.inf and got[0x7B] == 57344.0


def _finite_codes(shape, seed, fmt):
    """Random codes of one element format without NaN / infinity codes."""
    c = inputs.random_codes(shape, seed).numpy()
    if fmt == "e5m2":
        special = ((c >> 2) & 0x1F) == 31
        c = np.where(special, c & 0x83, c)     # exponent 31 -> 0: a subnormal of the same sign
    else:
        c = np.where((c & 0x7F) == 0x7F, c & 0xF8, c)
    return c.astype(np.uint8)


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_bruteforce_element_formats(a_fmt, b_fmt):
    """The other element-format pairs (the pages' E5M2E5M2, E4M3E5M2, E5M2E4M3
    kernel entries) against exact rationals, scales spread widely."""
    R, M, N, ka = 2, 3, 4, 64
    K = R * ka
    A = _finite_codes((M, K), 31, a_fmt)
    B = _finite_codes((N, K), 32, b_fmt)
    sA = inputs.random_scales((M, K // 32), 33, 40, 200).numpy()
    sB = inputs.random_scales((N, K // 32), 34, 40, 200).numpy()
    As, Ss = _split(A, sA, R, ka)
    got = oracle.gemm(As, Ss, B, sB, a_fmt=a_fmt, b_fmt=b_fmt)
    want = _exact.exact_gemm_fraction(As, Ss, B, sB, a_fmt=a_fmt, b_fmt=b_fmt)
    assert np.array_equal(got, want)


def test_e5m2_infinities_follow_ieee():
    """E5M2 infinities: inf x finite = inf, inf x 0 = NaN, +inf + -inf = NaN,
    checked against a float64 dot product (IEEE) of the decoded values."""
    R, M, N, ka = 1, 5, 3, 64
    K = R * ka
    A = np.full((M, K), 0x3C, np.uint8)        # 1.0
    B = np.full((N, K), 0x3C, np.uint8)
    A[0, 0] = 0x7C                               # +inf in block 0
    A[1, 0] = 0xFC                               # -inf
    A[2, 0] = 0x7C; A[2, 40] = 0xFC              # +inf and -inf in different blocks
    A[3, 5] = 0x7C
    B[1, 5] = 0x00                               # ... times +0 in column 1
    A[4, 7] = 0x7E                               # NaN code
    sA = np.full((M, K // 32), 127, np.uint8)
    sB = np.full((N, K // 32), 127, np.uint8)
    got = oracle.gemm([A], [sA], B, sB, a_fmt="e5m2", b_fmt="e5m2")
    with np.errstate(invalid="ignore"):
        ref = _exact.e5m2_values(A) @ _exact.e5m2_values(B).T
        want = np.where(np.isnan(ref), 0x7FC0, np.where(np.isinf(ref), np.where(ref > 0, 0x7F80, 0xFF80),
                                                       _exact.round_f64_to_bf16(np.nan_to_num(ref))))
    assert np.array_equal(got, want.astype(np.uint16)), (got, want)


def test_mixed_formats_identity_B():
    """E4M3 A times an E5M2 identity (1.0 = 0x3C) returns A exactly, and
    E5M2 A times an E4M3 identity (0x38) too."""
    M, K = 8, 64
    for a_fmt, b_fmt, one in (("e4m3", "e5m2", 0x3C), ("e5m2", "e4m3", 0x38)):
        A = _finite_codes((M, K), 41, a_fmt)
        B = np.zeros((K, K), np.uint8)
        np.fill_diagonal(B, one)
        sA = np.full((M, K // 32), 127, np.uint8)
        sB = np.full((K, K // 32), 127, np.uint8)
        got = oracle.gemm([A], [sA], B, sB, a_fmt=a_fmt, b_fmt=b_fmt)
        want = _exact.round_f64_to_bf16(_exact.values_of(A, a_fmt))
        assert np.array_equal(got, want), (a_fmt, b_fmt)


def test_round_bf16_random_vs_grid():
    rng = random.Random(7)
    for _ in range(3000):
        nd = rng.randint(1, 4)
        digits = [rng.randrange(1 << 31) for _ in range(nd)]
        exp0 = rng.randint(-272, 239 - 31 * (nd - 1))     # the oracle's exact range
        neg = rng.random() < 0.5
        x = sum(Fraction(d) * Fraction(2) ** (exp0 + 31 * i) for i, d in enumerate(digits))
        if neg:
            x = -x
        assert oracle.round_bf16(neg, digits, exp0) == _exact.round_fraction_to_bf16(x), (digits, exp0)


def test_round_bf16_ties_subnormals_overflow():
    # exact midpoints between neighbours, at several binades including subnormals
    cases = []
    for e in (-140, -134, -133, -127, -126, -20, 0, 7, 100, 119):
        for q in (128, 129, 200, 255):           # significand q * 2^(e-7) -> midpoint + half
            cases.append((2 * q + 1, e - 8))
    for mant, exp0 in cases:
        x = Fraction(mant) * Fraction(2) ** exp0
        got = oracle.round_bf16(False, [mant], exp0)
        assert got == _exact.round_fraction_to_bf16(x), (mant, exp0)
    # largest finite and the overflow threshold (ties to even goes to infinity)
    assert oracle.round_bf16(False, [255], 120) == 0x7F7F
    assert oracle.round_bf16(False, [511], 119) == 0x7F80
    assert oracle.round_bf16(False, [1], -134) == 0x0000       # half of min subnormal: tie to 0
    assert oracle.round_bf16(False, [3], -135) == 0x0001       # 0.75 min subnormal
    assert oracle.round_bf16(True, [1], -133) == 0x8001


# --- brute force on tiny inputs with exact rationals ----------------------------------

@pytest.mark.parametrize("R,M,N,ka,seed", [
    (1, 2, 3, 32, 0), (2, 3, 2, 32, 1), (3, 2, 4, 64, 2), (2, 4, 4, 64, 3), (3, 1, 1, 32, 4)])
def test_bruteforce_exact_rationals(R, M, N, ka, seed):
    K = R * ka
    A = inputs.random_codes((M, K), seed).numpy()
    B = inputs.random_codes((N, K), seed + 100).numpy()
    # wide scale spread, including extreme bytes; keep every output within range
    sA = inputs.random_scales((M, K // 32), seed + 200, 60, 190).numpy()
    sB = inputs.random_scales((N, K // 32), seed + 300, 60, 190).numpy()
    As, Ss = _split(A, sA, R, ka)
    got = oracle.gemm(As, Ss, B, sB)
    want = _exact.exact_gemm_fraction(As, Ss, B, sB)
    assert np.array_equal(got, want)


def test_bruteforce_cancellation_and_underflow():
    # blocks of opposite sign and very different scales: the sum must be exact
    R, M, N, ka = 2, 2, 2, 32
    K = R * ka
    A = np.zeros((M, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    A[:, 0] = 0x7E; A[:, 32] = 0xFE; A[:, 33] = 0x01     # 448, -448, 2^-9
    B[:, 0] = 0x38; B[:, 32] = 0x38; B[:, 33] = 0x38
    sA = np.full((M, K // 32), 127, np.uint8)
    sB = np.full((N, K // 32), 127, np.uint8)
    sA[1, 1] = 3                                            # second segment scaled by 2^-124
    As, Ss = _split(A, sA, R, ka)
    got = oracle.gemm(As, Ss, B, sB)
    want = _exact.exact_gemm_fraction(As, Ss, B, sB)
    assert np.array_equal(got, want)
    assert got[0, 0] == 0x3B00                              # 448 - 448 + 2^-9 = 2^-9


# --- unit scales: a float64 matmul is exact here ----------------------------------------

def test_unit_scales_equal_float64_matmul():
    R, M, N, ka = 3, 24, 40, 128
    K = R * ka
    A = inputs.random_codes((M, K), 11).numpy()
    B = inputs.random_codes((N, K), 12).numpy()
    sA = np.full((M, K // 32), 127, np.uint8)
    sB = np.full((N, K // 32), 127, np.uint8)
    # every product is a multiple of 2^-18 below 2^18 in size: K of them sum
    # exactly in float64 in any order
    ref = _exact.e4m3_values(A) @ _exact.e4m3_values(B).T
    want = _exact.round_f64_to_bf16(ref)
    As, Ss = _split(A, sA, R, ka)
    got = oracle.gemm(As, Ss, B, sB)
    assert np.array_equal(got, want)


# --- identity and one-hot B ----------------------------------------------------------------

def test_identity_B_returns_A():
    R, M, ka = 2, 16, 64
    K = N = R * ka
    A = inputs.random_codes((M, K), 21).numpy()
    sA = inputs.random_scales((M, K // 32), 22, 110, 140).numpy()
    B = np.zeros((N, K), np.uint8)
    B[np.arange(N), np.arange(K)] = 0x38                    # 1.0
    sB = np.full((N, K // 32), 127, np.uint8)
    As, Ss = _split(A, sA, R, ka)
    got = oracle.gemm(As, Ss, B, sB)
    vals = _exact.e4m3_values(A) * np.repeat(_exact.e8m0_values(sA), 32, axis=1)
    want = torch.from_numpy(vals).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # code 0x80 is -0; a sum that also holds +0 products is +0
    want = np.where(want == 0x8000, np.uint16(0), want)
    assert np.array_equal(got, want)


def test_one_hot_B_selects_columns():
    R, M, ka, N = 3, 8, 32, 20
    K = R * ka
    rng = np.random.default_rng(5)
    perm = rng.integers(0, K, size=N)
    A = inputs.random_codes((M, K), 31).numpy()
    sA = inputs.random_scales((M, K // 32), 32, 115, 135).numpy()
    B = np.zeros((N, K), np.uint8)
    B[np.arange(N), perm] = 0x38
    sB = np.full((N, K // 32), 127, np.uint8)
    As, Ss = _split(A, sA, R, ka)
    got = oracle.gemm(As, Ss, B, sB)
    vals = _exact.e4m3_values(A) * np.repeat(_exact.e8m0_values(sA), 32, axis=1)
    want = _exact.round_f64_to_bf16(vals[:, perm])
    assert np.array_equal(got, want)


# --- invariances ------------------------------------------------------------------------------

@pytest.mark.parametrize("d", [-5, 3])
def test_power_of_two_scale_invariance(d):
    w = inputs.Workload("pin", 2, 16, 64, 24, 16, 2, 41)
    x = inputs.make_inputs(w)
    A = [a.numpy() for a in x["A_seg"]]
    S = [s.numpy() for s in x["A_scale_seg"]]
    B, sB = x["B"].numpy(), x["B_scale"].numpy()
    base = oracle.gemm(A, S, B, sB)
    S2 = [(s.astype(np.int32) + d).astype(np.uint8) for s in S]
    shifted = oracle.gemm(A, S2, B, sB)
    f = oracle.bf16_bits_to_f32(base).astype(np.float64) * 2.0 ** d
    assert np.array_equal(shifted, _exact.round_f64_to_bf16(f))
    # the same through B's scales
    sB2 = (sB.astype(np.int32) + d).astype(np.uint8)
    assert np.array_equal(oracle.gemm(A, S, B, sB2), shifted)


def test_segment_permutation_invariance():
    w = inputs.Workload("pin", 4, 8, 64, 12, 8, 2, 43)
    x = inputs.make_inputs(w)
    A = [a.numpy() for a in x["A_seg"]]
    S = [s.numpy() for s in x["A_scale_seg"]]
    B, sB = x["B"].numpy(), x["B_scale"].numpy()
    ka = w.kPerRank
    sigma = [2, 0, 3, 1]
    A2 = [A[s] for s in sigma]
    S2 = [S[s] for s in sigma]
    B2 = np.concatenate([B[:, s * ka:(s + 1) * ka] for s in sigma], axis=1)
    sB2 = np.concatenate([sB[:, s * ka // 32:(s + 1) * ka // 32] for s in sigma], axis=1)
    assert np.array_equal(oracle.gemm(A, S, B, sB), oracle.gemm(A2, S2, B2, sB2))


def test_zero_A_gives_positive_zero():
    R, M, ka, N = 2, 4, 32, 4
    A = [np.zeros((M, ka), np.uint8) for _ in range(R)]
    S = [np.full((M, ka // 32), 127, np.uint8) for _ in range(R)]
    B = inputs.random_codes((N, R * ka), 3).numpy()
    sB = np.full((N, R * ka // 32), 127, np.uint8)
    assert np.all(oracle.gemm(A, S, B, sB) == 0)


def test_nan_codes_propagate_to_their_row_only():
    R, M, ka, N = 2, 3, 32, 2
    A = [np.full((M, ka), 0x38, np.uint8) for _ in range(R)]
    A[1][1, 5] = 0x7F
    S = [np.full((M, ka // 32), 127, np.uint8) for _ in range(R)]
    B = np.full((N, R * ka), 0x38, np.uint8)
    sB = np.full((N, R * ka // 32), 127, np.uint8)
    C = oracle.gemm(A, S, B, sB)
    assert np.all(C[1] == 0x7FC0)
    assert np.all(C[[0, 2]] == 0x4280)                      # 64.0


def test_row_col_subsets_match_full():
    w = inputs.Workload("pin", 2, 16, 64, 24, 16, 2, 45)
    x = inputs.make_inputs(w)
    full = oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"])
    rows, cols = [3, 0, 15], [23, 1, 7, 7]
    sub = oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"], rows=rows, cols=cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])


# --- hand-worked fixtures ---------------------------------------------------------------------

def _load_fixture(path):
    with open(path) as f:
        fx = json.load(f)
    R, M, ka, N = fx["R"], fx["M"], fx["kPerRank"], fx["N"]
    K = R * ka
    A = np.zeros((M, K), np.uint8)
    for k, c in fx["A_codes"].items():
        A[0, int(k)] = c
    B = np.zeros((N, K), np.uint8)
    for key, c in fx["B_codes"].items():
        n, k = (int(v) for v in key.split(","))
        B[n, k] = c
    sA = np.array(fx["A_scales"], np.uint8).reshape(R, M, ka // 32)
    sB = np.array(fx["B_scales"], np.uint8)
    As = [np.ascontiguousarray(A[:, r * ka:(r + 1) * ka]) for r in range(R)]
    Ss = [np.ascontiguousarray(sA[r]) for r in range(R)]
    return fx, As, Ss, B, sB


def test_golden_handworked_fixtures():
    gdir = os.path.join(HERE, "golden")
    files = sorted(f for f in os.listdir(gdir) if f.startswith("handworked") and f.endswith(".json"))
    assert files
    for name in files:
        fx, As, Ss, B, sB = _load_fixture(os.path.join(gdir, name))
        got = oracle.gemm(As, Ss, B, sB)
        assert got.ravel().tolist() == fx["C_bf16_bits"], name


# --- the pins catch planted mistakes ----------------------------------------------------------

MUTANTS = {
    "drop_last_block": ("for (int64_t b = 0; b < nb; ++b) {\n                if (Anan[b]",
                        "for (int64_t b = 0; b < nb - 1; ++b) {\n                if (Anan[b]"),
    "scale_bias_off": ("int shift = (sa - 127) + (sb - 127) - 18 - UNIT_EXP;",
                       "int shift = (sa - 126) + (sb - 127) - 18 - UNIT_EXP;"),
    "segment_offset": ("Au[r * j->ka + k] = e4m3_units(src[k], &nan);",
                       "Au[((r + 1) % j->R) * j->ka + k] = e4m3_units(src[k], &nan);"),
    "ties_away": ("if (round_bit && (sticky || (q & 1u))) q += 1;",
                  "if (round_bit) q += 1;"),
    "sign_dropped": ("else big_add_shifted(&neg, (uint64_t)(-s), shift);",
                     "else big_add_shifted(&pos, (uint64_t)(-s), shift);"),
    "subnormal_decode": ("if (e == 0) mag = m;", "if (e == 0) mag = 2 * m;"),
    "e5m2_exponent_bias": ("else mag = (int64_t)(4 + m) << (e - 1);", "else mag = (int64_t)(4 + m) << e;"),
    "e5m2_wide_units": ("int shift = (sa - 127) + (sb - 127) - 32 - UNIT_EXP;",
                        "int shift = (sa - 127) + (sb - 127) - 25 - UNIT_EXP;"),
    "mixed_units": ("shift -= j->uexp_fix;", "shift += j->uexp_fix;"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mxa2a_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    csrc = tmp_path / "mutant.c"
    csrc.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-D_DEFAULT_SOURCE", "-shared", "-fPIC",
                           "-pthread", "-o", str(so), str(csrc)])
    lib = ctypes.CDLL(str(so))
    good = oracle._load()
    for fn in ("mxa2a_oracle_gemm", "mxa2a_oracle_gemm_fmt", "mxa2a_oracle_round_bf16",
               "mxa2a_oracle_decode_e4m3", "mxa2a_oracle_decode_e5m2", "mxa2a_oracle_decode_e8m0"):
        getattr(lib, fn).argtypes = getattr(good, fn).argtypes
        getattr(lib, fn).restype = getattr(good, fn).restype

    saved = oracle._lib
    oracle._lib = lib
    failures = 0
    try:
        for check in (lambda: test_bruteforce_exact_rationals(2, 3, 2, 32, 1),
                      lambda: test_bruteforce_exact_rationals(3, 2, 4, 64, 2),
                      test_golden_handworked_fixtures,
                      test_round_bf16_ties_subnormals_overflow,
                      test_one_hot_B_selects_columns,
                      test_unit_scales_equal_float64_matmul,
                      test_e5m2_decode_exhaustive_vs_torch,
                      lambda: test_bruteforce_element_formats("e5m2", "e5m2"),
                      lambda: test_bruteforce_element_formats("e4m3", "e5m2")):
            try:
                check()
            except AssertionError:
                failures += 1
    finally:
        oracle._lib = saved
    assert failures > 0, f"mutant {name} survived every pin"
