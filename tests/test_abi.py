"""The C-ABI library: builds, loads, exports every declared symbol, host-side rules.

No compute call is made here (no GPU is needed): only symbol presence, the
pure-host shape validation, error strings and the binding's constants.
"""
import ctypes
import os
import re

import pytest

from all_mxfp8_block_gb300 import build as mxbuild
from all_mxfp8_block_gb300 import mxa2a

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxa2a.h")


@pytest.fixture(scope="module")
def lib():
    mxbuild.build()
    return ctypes.CDLL(mxbuild.LIB)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(mxa2a_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def declared_constants():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {k: int(v) for k, v in re.findall(r"\b(MXA2A_[A-Z_0-9]+)\s*=\s*(\d+)", src)}


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_header():
    names = declared_functions()
    for n in names:
        assert callable(getattr(mxa2a, n)), n
    bound = {s[0] for s in mxa2a._SIGS}
    assert set(names) == bound


def test_binding_constants_match_header():
    consts = declared_constants()
    assert consts
    for k, v in consts.items():
        assert getattr(mxa2a, k) == v, k


def test_validate_shape_rules(lib):
    v = mxa2a.mxa2a_validate
    ok, bad = mxa2a.MXA2A_OK, mxa2a.MXA2A_ERR_INVALID_SHAPE
    # the five workloads
    assert v(2, 128, 128, 256, 64, 2) == ok
    assert v(4, 2048, 1024, 4096, 256, 2) == ok
    assert v(8, 4096, 896, 2048, 512, 4) == ok
    assert v(8, 8192, 1024, 8192, 512, 4) == ok
    assert v(16, 64, 512, 7168, 64, 2) == ok
    # rules
    assert v(0, 128, 128, 256, 64, 2) == bad            # R >= 1
    assert v(65, 128, 128, 256, 64, 2) == bad           # R <= 64
    assert v(2, 128, 96, 256, 64, 2) == bad             # kPerRank % 128
    assert v(2, 128, 128, 250, 64, 2) == bad            # N % 16
    assert v(2, 128, 128, 256, 96, 2) == bad            # commMSize % 64
    assert v(2, 192, 128, 256, 128, 2) == bad           # M % commMSize
    assert v(2, 128, 128, 256, 64, 0) == bad            # buffer_num >= 1
    assert v(2, 128, 128, 256, 64, 9) == bad            # buffer_num <= 8
    assert v(2, 128, 128, 256, 64, 1) == bad            # a 128-row tile spans 2 steps of 64 rows
    assert v(2, 256, 128, 256, 128, 1) == ok            # one step per tile: a single slot suffices
    assert v(2, 384, 128, 256, 192, 1) == bad           # 192-row steps: tiles straddle steps
    assert v(2, 384, 128, 256, 192, 2) == ok
    assert v(1, 1 << 21, 128, 256, 64, 2) == bad        # size limit


def test_strerror(lib):
    assert mxa2a.strerror(0) == "ok"
    assert "timed out" in mxa2a.strerror(mxa2a.MXA2A_ERR_TIMEOUT)
    assert mxa2a.strerror(12345) == "unknown error"


def test_null_plan_calls_fail_cleanly(lib):
    assert mxa2a.load().mxa2a_set_option(None, mxa2a.MXA2A_OPT_ZIGZAG, 1) == mxa2a.MXA2A_ERR_NULL_PTR
    assert mxa2a.load().mxa2a_run(None, None, None, None, None, None, None) == mxa2a.MXA2A_ERR_NULL_PTR
    mxa2a.load().mxa2a_destroy(None)


def test_validate_allgather_rules(lib):
    v = mxa2a.mxa2a_validate_allgather
    ok, bad = mxa2a.MXA2A_OK, mxa2a.MXA2A_ERR_INVALID_SHAPE
    assert v(4, 512, 4096, 4096, 256, 2) == ok
    assert v(1, 128, 256, 256, 64, 2) == ok
    assert v(0, 512, 4096, 4096, 256, 2) == bad          # R >= 1
    assert v(65, 64, 256, 256, 64, 2) == bad            # R <= 64
    assert v(4, 320, 4096, 4096, 256, 2) == bad         # rowsPerRank % commMSize
    assert v(4, 512, 4000, 4096, 256, 2) == bad         # K % 128
    assert v(4, 512, 4096, 4096, 96, 2) == bad          # commMSize % 64
    assert v(1 << 10, 1 << 11, 256, 256, 64, 2) == bad  # R > 64 (and M > 2^20)
    assert v(64, 1 << 15, 256, 256, 64, 2) == bad       # M = R * rowsPerRank > 2^20


def test_validate_reduce_scatter_rules(lib):
    v = mxa2a.mxa2a_validate_reduce_scatter
    ok, bad = mxa2a.MXA2A_OK, mxa2a.MXA2A_ERR_INVALID_SHAPE
    assert v(4, 1, 2048, 4096, 4096) == ok
    assert v(1, 0, 64, 128, 16) == ok
    assert v(4, 4, 2048, 4096, 4096) == bad             # rank < R
    assert v(4, -1, 2048, 4096, 4096) == bad            # rank >= 0
    assert v(4, 0, 2048 + 64, 4096, 4096) == bad        # M % (64 R)
    assert v(4, 0, 128, 4096, 4096) == bad              # M >= 64 R
    assert v(4, 0, 2048, 4000, 4096) == bad             # K % 128
    assert v(4, 0, 2048, 4096, 4008) == bad             # N % 16
    assert v(65, 0, 65 * 64, 128, 16) == bad            # R <= 64


def test_null_sibling_calls_fail_cleanly(lib):
    L = mxa2a.load()
    assert L.mxa2a_run_reduce_scatter(None, None, None, None, None, None, None, None, None) == \
        mxa2a.MXA2A_ERR_NULL_PTR
    assert L.mxa2a_run_reduce_scatter_unfused(None, None, None, None, None, None, None, None, None) == \
        mxa2a.MXA2A_ERR_NULL_PTR


def test_validate_allreduce_rules(lib):
    v = mxa2a.mxa2a_validate_allreduce
    ok, bad = mxa2a.MXA2A_OK, mxa2a.MXA2A_ERR_INVALID_SHAPE
    assert v(4, 1, 2048, 4096, 4096) == ok
    assert v(1, 0, 64, 128, 16) == ok
    assert v(3, 1, 192, 384, 272) == ok
    assert v(4, 4, 2048, 4096, 4096) == bad             # rank < R
    assert v(0, 0, 2048, 4096, 4096) == bad             # R >= 1
    assert v(4, 0, 2048 + 32, 4096, 4096) == bad        # M % 64
    assert v(4, 0, 2048, 4000, 4096) == bad             # K % 128
    assert v(4, 0, 2048, 4096, 4008) == bad             # N % 16
    L = mxa2a.load()
    assert L.mxa2a_run_allreduce(None, None, None, None, None, None, None, None, None) == mxa2a.MXA2A_ERR_NULL_PTR
