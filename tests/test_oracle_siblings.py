"""Pins of the sibling-operator oracle functions (AllGather + GEMM, GEMM +
ReduceScatter, GEMM + AllReduce; the performance optimisation guide, section 3) and of its
float64 -> BF16 rounding, against things other than the oracle itself:
torch's BF16 conversion, the explicit BF16 grid of ``tests/_exact.py``, exact
rational sums, and identity operands whose products are known block by block.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from all_mxfp8_block_gb300 import inputs
from tests import _exact as X


def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


# --- float64 -> BF16 ------------------------------------------------------------------

def test_round_f64_to_bf16_matches_torch_on_float32_values():
    """Random float32 values over the whole range (subnormals, overflow) and
    every tie between BF16 neighbours in a few binades: torch rounds float32
    to BF16 to nearest even, and float32 values are exact in float64."""
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    got = oracle.round_f64_to_bf16(x.astype(np.float64))
    want = _torch_bf16_bits(x)
    assert np.array_equal(got, want)
    # ties: the midpoint of BF16 neighbours (9 significant bits, exact in float32)
    lo = np.arange(0x3F00, 0x4100, dtype=np.uint32)
    vlo = (lo << 16).view(np.float32).astype(np.float64)
    vhi = ((lo + 1) << 16).view(np.float32).astype(np.float64)
    mid = (vlo + vhi) / 2
    for sign in (1.0, -1.0):
        assert np.array_equal(oracle.round_f64_to_bf16(sign * mid), _torch_bf16_bits((sign * mid).astype(np.float32)))


def test_round_f64_to_bf16_beyond_float32_against_the_grid():
    """float64 values that float32 cannot hold (just off a tie, far below the
    smallest subnormal, past the largest finite) against the exact grid search."""
    rng = np.random.default_rng(6)
    base = rng.uniform(-4, 4, size=5000) * 2.0 ** rng.integers(-140, 128, size=5000)
    nudge = base * (1 + rng.choice([-1, 1], size=5000) * 2.0 ** -40)
    ties = (np.array([1.0, 3.0, 0.75]) + 2.0 ** -8) * (1 + 2.0 ** -45)      # just above a tie
    vals = np.concatenate([base, nudge, ties, -ties, [2.0 ** -134, 2.0 ** -133 * 1.5, 3.3e38, 3.4e38]])
    got = oracle.round_f64_to_bf16(vals)
    want = X.round_f64_to_bf16(vals)
    assert np.array_equal(got, want)
    f = oracle.round_f64_to_bf16(np.array([np.inf, -np.inf, np.nan]))
    assert f[0] == 0x7F80 and f[1] == 0xFF80 and (f[2] & 0x7F80) == 0x7F80 and (f[2] & 0x7F) != 0


# --- AllGather + GEMM ---------------------------------------------------------------------

def _identity_b(n: int):
    """B = I (E4M3 1.0 = 0x38 on the diagonal), unit scales: C = the scaled A."""
    B = np.zeros((n, n), dtype=np.uint8)
    np.fill_diagonal(B, 0x38)
    return B, np.full((n, n // 32), 127, dtype=np.uint8)


def _finite_codes(shape, seed):
    c = inputs.random_codes(shape, seed).numpy()
    return c


def test_allgather_identity_B_stacks_blocks_in_rank_order():
    """With B = I the product is the gathered A itself: block j of the result
    is block j's decoded, scaled rows (values exact in BF16 for scales near
    2^0), so a wrong block order or row offset shows at once."""
    R, rows, K = 3, 64, 128
    A = [_finite_codes((rows, K), 40 + j) for j in range(R)]
    S = [inputs.random_scales((rows, K // 32), 50 + j, lo=117, hi=137).numpy() for j in range(R)]
    B, Bs = _identity_b(K)
    C = oracle.gemm_allgather(A, S, B, Bs)
    assert C.shape == (R * rows, K)
    for j in range(R):
        want = X.e4m3_values(A[j]) * np.repeat(X.e8m0_values(S[j]), 32, axis=1)
        assert np.array_equal(C[j * rows:(j + 1) * rows], X.round_f64_to_bf16(want)), f"block {j}"
    # a sub-block request gives the same bits
    rs, cs = [5, 64, 190], [0, 31, 127]
    assert np.array_equal(oracle.gemm_allgather(A, S, B, Bs, rows=rs, cols=cs), C[np.ix_(rs, cs)])


def test_allgather_brute_force_tiny():
    """Exact rational brute force on a tiny gather (3 blocks of 2 rows, K 64)."""
    R, rows, K, N = 3, 2, 64, 5
    A = [_finite_codes((rows, K), 60 + j) for j in range(R)]
    S = [inputs.random_scales((rows, K // 32), 70 + j, lo=120, hi=134).numpy() for j in range(R)]
    B = _finite_codes((N, K), 80)
    Bs = inputs.random_scales((N, K // 32), 81, lo=120, hi=134).numpy()
    want = X.exact_gemm_fraction([np.concatenate(A, axis=0)], [np.concatenate(S, axis=0)], B, Bs)
    assert np.array_equal(oracle.gemm_allgather(A, S, B, Bs), want)


# --- GEMM + ReduceScatter -------------------------------------------------------------

def _rs_identity_case(R, rank, rows=64, K=128, seed=0):
    M = R * rows
    A = _finite_codes((M, K), 90 + seed)
    S = inputs.random_scales((M, K // 32), 91 + seed, lo=117, hi=137).numpy()
    B, Bs = _identity_b(K)
    rng = np.random.default_rng(92 + seed)
    recv = [None if j == rank else
            _torch_bf16_bits(rng.standard_normal((rows, K)).astype(np.float32) * 4) for j in range(R)]
    return A, S, B, Bs, recv


@pytest.mark.parametrize("R,rank", [(3, 0), (3, 1), (3, 2), (4, 3)])
def test_reduce_scatter_identity_B_blocks_and_exact_sum(R, rank):
    """B = I: this rank's partial is its decoded, scaled A.  Block j != rank
    must be sent as is; the output is the exact rational sum of this rank's
    block and the R-1 received partials, rounded once to BF16 (grid search)."""
    rows, K = 64, 128
    A, S, B, Bs, recv = _rs_identity_case(R, rank, rows, K, seed=R + rank)
    send, out = oracle.gemm_reduce_scatter(A, S, B, Bs, recv, R, rank)
    P = X.round_f64_to_bf16(X.e4m3_values(A) * np.repeat(X.e8m0_values(S), 32, axis=1))
    assert sorted(send) == [j for j in range(R) if j != rank]
    for j, blk in send.items():
        assert np.array_equal(blk, P[j * rows:(j + 1) * rows]), f"send block {j}"
    own = P[rank * rows:(rank + 1) * rows]
    parts = [own if j == rank else recv[j] for j in range(R)]
    vals = [(p.astype(np.uint32) << 16).view(np.float32) for p in parts]
    want = np.zeros((rows, K), dtype=np.uint16)
    for i in range(rows):
        for n in range(K):
            want[i, n] = X.round_fraction_to_bf16(sum(Fraction(float(v[i, n])) for v in vals))
    assert np.array_equal(out, want)


def test_reduce_scatter_single_rank_is_the_gemm():
    """R = 1: nothing to send or receive, the output is the plain product."""
    A = _finite_codes((64, 128), 100)
    S = inputs.random_scales((64, 4), 101, lo=120, hi=134).numpy()
    B = _finite_codes((48, 128), 102)
    Bs = inputs.random_scales((48, 4), 103, lo=120, hi=134).numpy()
    send, out = oracle.gemm_reduce_scatter(A, S, B, Bs, [None], 1, 0)
    assert send == {}
    assert np.array_equal(out, oracle.gemm([A], [S], B, Bs))
    assert np.array_equal(out[:3], X.exact_gemm_fraction([A[:3]], [S[:3]], B, Bs))


def test_reduce_scatter_cancellation_is_exact():
    """Received partials that cancel this rank's block exactly give +0, and
    two small partials whose sum crosses a rounding midpoint that neither
    crosses alone are rounded once, after the exact sum (not per addition)."""
    R, rank, rows, K = 2, 0, 64, 128
    A, S, B, Bs, _ = _rs_identity_case(R, rank, rows, K, seed=7)
    P = X.round_f64_to_bf16(X.e4m3_values(A) * np.repeat(X.e8m0_values(S), 32, axis=1))
    neg = P[:rows] ^ np.uint16(0x8000)
    _, out = oracle.gemm_reduce_scatter(A, S, B, Bs, [None, neg], R, rank)
    assert np.all((out == 0) | (out == 0x8000))
    # three ranks, this rank's partial exactly 1.0 (A = 1.0 codes, B = I) and two
    # received 3 * 2^-10: the exact sum 1 + 6 * 2^-10 is past the midpoint to
    # 1 + 2^-7, while rounding after each addition would stay at 1.0
    R, rank = 3, 0
    A1 = np.full((R * rows, K), 0x38, dtype=np.uint8)
    S1 = np.full((R * rows, K // 32), 127, dtype=np.uint8)
    d = _torch_bf16_bits(np.full((rows, K), 3 * 2.0 ** -10, dtype=np.float32))
    send, out = oracle.gemm_reduce_scatter(A1, S1, B, Bs, [None, d, d], R, rank)
    assert np.all(out == 0x3F81)
    assert all(np.all(v == 0x3F80) for v in send.values())


def test_exact_sum_refuses_an_inexact_float64_sum():
    with pytest.raises(AssertionError):
        oracle._exact_sum([np.array([1.0]), np.array([2.0 ** -60])])


# --- GEMM + AllReduce (one-shot) -----------------------------------------------------

@pytest.mark.parametrize("R,rank", [(3, 0), (3, 2), (2, 1)])
def test_allreduce_identity_B_publishes_and_sums_every_row(R, rank):
    """B = I: the published partial is the decoded, scaled A; the output is,
    for every row, the exact rational sum of that and the R-1 peers'
    partials, rounded once to BF16 (grid search)."""
    M, K = 64, 128
    A = _finite_codes((M, K), 120 + R + rank)
    S = inputs.random_scales((M, K // 32), 121, lo=117, hi=137).numpy()
    B, Bs = _identity_b(K)
    rng = np.random.default_rng(122 + rank)
    recv = [None if j == rank else
            _torch_bf16_bits(rng.standard_normal((M, K)).astype(np.float32) * 4) for j in range(R)]
    pub, out = oracle.gemm_allreduce(A, S, B, Bs, recv, R, rank)
    P = X.round_f64_to_bf16(X.e4m3_values(A) * np.repeat(X.e8m0_values(S), 32, axis=1))
    assert np.array_equal(pub, P)
    vals = [(p.astype(np.uint32) << 16).view(np.float32) for p in (P if j == rank else recv[j] for j in range(R))]
    want = np.zeros((M, K), dtype=np.uint16)
    for i in range(M):
        for n in range(K):
            want[i, n] = X.round_fraction_to_bf16(sum(Fraction(float(v[i, n])) for v in vals))
    assert np.array_equal(out, want)


def test_allreduce_is_the_reduce_scatter_of_one_block():
    """Every rank's all-reduce output equals the reduce-scatter's output
    blocks stacked: block j of the all-reduce is what rank j's reduce-scatter
    computes from the same partials."""
    R, M, K = 3, 192, 128
    A = _finite_codes((M, K), 130)
    S = inputs.random_scales((M, K // 32), 131, lo=120, hi=134).numpy()
    B, Bs = _identity_b(K)
    rng = np.random.default_rng(132)
    rank = 1
    recv = [None if j == rank else
            _torch_bf16_bits(rng.standard_normal((M, K)).astype(np.float32)) for j in range(R)]
    _, out = oracle.gemm_allreduce(A, S, B, Bs, recv, R, rank)
    rows = M // R
    _, rs_out = oracle.gemm_reduce_scatter(A, S, B, Bs, [None if r is None else r[rank * rows:(rank + 1) * rows]
                                                        for r in recv], R, rank)
    assert np.array_equal(out[rank * rows:(rank + 1) * rows], rs_out)
