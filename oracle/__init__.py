"""CPU oracle for the fused AllToAll + MXFP8 block-scaled GEMM.

TEST INFRASTRUCTURE ONLY.  The exact reference the CUDA path is checked
against: only ``tests/``, the package's ``smoke()`` check and the benchmark's
CPU-baseline leg may import it.  The CUDA library and its Python binding never
import, link or call anything here, and nothing here uses them.

The arithmetic lives in ``mxa2a_oracle.c`` (plain C, exact integer
accumulation, one rounding to BF16); this module builds it with ``gcc`` on
first use and marshals arguments through ``ctypes``.

Every oracle function is pinned by tests in ``tests/test_oracle_pins.py``
against things other than itself: torch's float8 decoders (exhaustive), exact
rational brute force, float64 matmul of exactly representable cases, identity
and one-hot operands, power-of-two scale invariance, segment-order
permutation and hand-worked fixtures in ``tests/golden/``.  The two sibling
fused operators (AllGather + GEMM, GEMM + ReduceScatter, GEMM + AllReduce,
the performance optimisation guide's section 3 cases) are compositions of
:func:`gemm` with a row stack and with an exact sum rounded once; they are pinned in
``tests/test_oracle_siblings.py`` (identity operands with known blocks, exact
rational sums, torch's BF16 rounding).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxa2a_oracle.c")
_LIB = os.path.join(_HERE, "libmxa2a_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmxa2a_oracle.so`` (host gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-shared",
                               "-fPIC", "-pthread", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.mxa2a_oracle_gemm.restype = ctypes.c_int
            lib.mxa2a_oracle_gemm.argtypes = [
                ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int]
            lib.mxa2a_oracle_gemm_fmt.restype = ctypes.c_int
            lib.mxa2a_oracle_gemm_fmt.argtypes = [
                ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_int]
            lib.mxa2a_oracle_decode_e5m2.restype = ctypes.c_double
            lib.mxa2a_oracle_decode_e5m2.argtypes = [ctypes.c_uint8]
            lib.mxa2a_oracle_decode_e4m3.restype = ctypes.c_double
            lib.mxa2a_oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
            lib.mxa2a_oracle_decode_e8m0.restype = ctypes.c_double
            lib.mxa2a_oracle_decode_e8m0.argtypes = [ctypes.c_uint8]
            lib.mxa2a_oracle_round_bf16.restype = ctypes.c_uint16
            lib.mxa2a_oracle_round_bf16.argtypes = [
                ctypes.c_int, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, ctypes.c_int]
            _lib = lib
    return _lib


def _np_u8(t) -> np.ndarray:
    a = t.numpy() if hasattr(t, "numpy") else np.asarray(t)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8, a.dtype
    return a


def decode_e4m3(code: int) -> float:
    """Value of one E4M3 ("fn") code; NaN for 0x7F / 0xFF."""
    return _load().mxa2a_oracle_decode_e4m3(code)


def decode_e5m2(code: int) -> float:
    """Value of one E5M2 code; +-inf for 0x7C / 0xFC, NaN for the other exponent-31 codes."""
    return _load().mxa2a_oracle_decode_e5m2(code)


def decode_e8m0(code: int) -> float:
    """Value 2^(code-127) of one E8M0 scale byte; NaN for 0xFF."""
    return _load().mxa2a_oracle_decode_e8m0(code)


def round_bf16(negative: bool, digits: list[int], exp0: int) -> int:
    """BF16 bits of ``(-1)^negative * sum_i digits[i] * 2^(exp0 + 31 i)``,
    rounded once to nearest, ties to even (digits < 2^31)."""
    arr = (ctypes.c_uint32 * max(1, len(digits)))(*digits)
    return int(_load().mxa2a_oracle_round_bf16(int(negative), arr, len(digits), exp0))


FORMATS = {"e4m3": 0, "e5m2": 1}


def gemm(A_seg, A_scale_seg, B, B_scale, rows=None, cols=None, nthreads: int = 0,
         a_fmt: str = "e4m3", b_fmt: str = "e4m3") -> np.ndarray:
    """Exact ``C = bf16(concat_r(A_r * sA_r) @ (B * sB)^T)`` as uint16 BF16 bits.

    ``A_seg[r]`` uint8 [M][ka], ``A_scale_seg[r]`` uint8 [M][ka/32],
    ``B`` uint8 [N][R*ka] (B stored transposed), ``B_scale`` uint8 [N][R*ka/32].
    ``rows`` / ``cols`` select a sub-block of C (default: all of it).
    ``a_fmt`` / ``b_fmt``: element format of A / B codes, "e4m3" or "e5m2"
    (the kernel entries E4M3E4M3, E5M2E5M2, E4M3E5M2, E5M2E4M3).
    """
    lib = _load()
    A = [_np_u8(a) for a in A_seg]
    S = [_np_u8(s) for s in A_scale_seg]
    Bn, Bs = _np_u8(B), _np_u8(B_scale)
    R = len(A)
    M, ka = A[0].shape
    N = Bn.shape[0]
    assert Bn.shape == (N, R * ka) and Bs.shape == (N, R * ka // 32)
    for a, s in zip(A, S):
        assert a.shape == (M, ka) and s.shape == (M, ka // 32)
    r_arr = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c_arr = None if cols is None else np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    nr = M if r_arr is None else len(r_arr)
    nc = N if c_arr is None else len(c_arr)
    out = np.zeros((nr, nc), dtype=np.uint16)
    a_ptrs = (ctypes.c_void_p * R)(*[a.ctypes.data for a in A])
    s_ptrs = (ctypes.c_void_p * R)(*[s.ctypes.data for s in S])
    rc = lib.mxa2a_oracle_gemm_fmt(
        R, M, ka, N, a_ptrs, s_ptrs, Bn.ctypes.data, Bs.ctypes.data, FORMATS[a_fmt], FORMATS[b_fmt],
        None if r_arr is None else r_arr.ctypes.data, nr,
        None if c_arr is None else c_arr.ctypes.data, nc,
        out.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle: bad arguments")
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_f64_to_bf16(x) -> np.ndarray:
    """BF16 bit patterns (uint16) of float64 values, rounded to nearest with
    ties to even.  BF16 keeps 8 significant bits; a finite x with
    2^e <= |x| < 2^(e+1) is rounded to a multiple of 2^(e-7), and below the
    smallest normal (2^-126) to a multiple of 2^-133 (the subnormal spacing).
    Dividing by that power of two is exact in float64 and ``np.rint`` rounds
    half to even, so the rounding is exact.  Magnitudes that round to 2^128 or
    beyond become infinities; NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, e = np.frexp(xf)                      # |x| = m 2^e, m in [0.5, 1): binade 2^(e-1)
    q = np.maximum(e - 1 - 7, -133)          # exponent of the BF16 spacing there
    r = np.rint(np.ldexp(xf, -q))            # exact scaling, ties to even
    out[finite] = np.ldexp(r, q)[finite]
    out[~finite] = x[~finite]
    out = np.where(np.abs(out) >= 2.0 ** 128, np.copysign(np.inf, out), out)
    f32 = out.astype(np.float32)             # exact: every BF16 value is a float32
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float64 (exact)."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def gemm_allgather(A_blk, A_scale_blk, B, B_scale, rows=None, cols=None, nthreads: int = 0,
                   a_fmt: str = "e4m3", b_fmt: str = "e4m3") -> np.ndarray:
    """AllGather + GEMM (performance optimisation guide, section 3.1, which
    names the operator only): the R row blocks ``A_blk[j]`` ([rowsPerRank][K]
    codes, scales [rowsPerRank][K/32]) are gathered, i.e. stacked along M with
    block j at rows j*rowsPerRank.., and multiplied by B exactly as
    :func:`gemm` does with a single K segment.  Returns BF16 bits [M][N] (or
    the ``rows`` x ``cols`` sub-block)."""
    A = np.concatenate([_np_u8(a) for a in A_blk], axis=0)
    S = np.concatenate([_np_u8(s) for s in A_scale_blk], axis=0)
    return gemm([A], [S], B, B_scale, rows=rows, cols=cols, nthreads=nthreads, a_fmt=a_fmt, b_fmt=b_fmt)


def _exact_sum(terms):
    """Sum float64 arrays in float64, asserting that no addition rounded
    (Knuth's two-sum error term is zero wherever the result is finite)."""
    s = np.zeros_like(terms[0])
    for t in terms:
        new = s + t
        bp = new - s
        err = (s - (new - bp)) + (t - bp)
        ok = ~np.isfinite(new) | (err == 0)
        assert np.all(ok), "oracle: the float64 sum is not exact for these inputs"
        s = new
    return s


def gemm_reduce_scatter(A, A_scale, B, B_scale, recv, R: int, rank: int, nthreads: int = 0,
                        a_fmt: str = "e4m3", b_fmt: str = "e4m3"):
    """GEMM + ReduceScatter from rank ``rank`` of ``R`` (performance
    optimisation guide, section 3.2, which names the operator only).  This
    rank's partial is P = :func:`gemm` of its A [M][K] and B [N][K], as BF16
    (the type the partials travel in).  Rows j*Mr .. (j+1)*Mr - 1 (Mr = M/R)
    of P are the block sent to rank j; this rank's output is the sum over
    ranks j of block ``rank`` of rank j's partial (``recv[j]``, BF16 bits
    [Mr][N], for j != rank; P's own block for j == rank), computed exactly and
    rounded once to BF16.  Returns ``(send, out)``: ``send`` a dict j -> BF16
    bits [Mr][N] for j != rank, ``out`` BF16 bits [Mr][N]."""
    P = gemm([A], [A_scale], B, B_scale, nthreads=nthreads, a_fmt=a_fmt, b_fmt=b_fmt)
    M = P.shape[0]
    assert M % R == 0 and 0 <= rank < R and len(recv) == R
    Mr = M // R
    send = {j: P[j * Mr:(j + 1) * Mr].copy() for j in range(R) if j != rank}
    terms = []
    for j in range(R):
        blk = P[rank * Mr:(rank + 1) * Mr] if j == rank else np.asarray(recv[j]).view(np.uint16)
        assert blk.shape == (Mr, P.shape[1])
        terms.append(bf16_bits_to_f64(blk))
    out = round_f64_to_bf16(_exact_sum(terms))
    return send, out


def gemm_allreduce(A, A_scale, B, B_scale, recv, R: int, rank: int, nthreads: int = 0,
                   a_fmt: str = "e4m3", b_fmt: str = "e4m3"):
    """GEMM + AllReduce, one-shot, from rank ``rank`` of ``R`` (performance
    optimisation guide, section 3.3, which names the operator only).  This
    rank's partial P = :func:`gemm` of its A [M][K] and B [N][K], as BF16, is
    published; its output is the sum over ranks j of rank j's partial
    (``recv[j]``, BF16 bits [M][N], for j != rank; P for j == rank), computed
    exactly and rounded once to BF16.  Returns ``(pub, out)``, both BF16 bits
    [M][N]."""
    P = gemm([A], [A_scale], B, B_scale, nthreads=nthreads, a_fmt=a_fmt, b_fmt=b_fmt)
    assert 0 <= rank < R and len(recv) == R
    terms = []
    for j in range(R):
        blk = P if j == rank else np.asarray(recv[j]).view(np.uint16)
        assert blk.shape == P.shape
        terms.append(bf16_bits_to_f64(blk))
    return P, round_f64_to_bf16(_exact_sum(terms))
