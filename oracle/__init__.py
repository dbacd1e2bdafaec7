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
permutation and hand-worked fixtures in ``tests/golden/``.
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
