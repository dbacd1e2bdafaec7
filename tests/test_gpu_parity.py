"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Gate per element: |gpu - ref| <= 1e-2 + 1e-2*|ref| (the pages' verify
tolerance, atol = rtol = 1e-2, measured against the exact oracle).  Small
shapes are compared in full; the full-size workloads on sampled rows (every
column), in the launch configuration the benchmark times.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from all_mxfp8_block_gb300 import inputs, mxa2a
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from all_mxfp8_block_gb300 import build
    build.build()
    mxa2a.load()
    torch.cuda.init()


def _plan(w, **opts):
    p = mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num)
    p.set_option(mxa2a.MXA2A_OPT_TIMEOUT_NS, opts.pop("timeout_ns", 500_000_000))
    for k, v in opts.items():
        p.set_option(getattr(mxa2a, "MXA2A_OPT_" + k.upper()), v)
    return p


def _status_ok(p):
    st = p.status()
    assert st["code"] == 0, st


def _check_full(w, fused=True, **opts):
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, **opts) as p:
        C = gu.run_gpu(p, d, w.M, w.N, fused=fused)
        torch.cuda.synchronize()
        _status_ok(p)
        got = gu.host_bits(C)
    ref = gu.oracle_full(x)
    gu.assert_parity(got, ref, f"{w.name} fused={fused} {opts}")
    return got, ref


# --- targeted layout checks: exact results ------------------------------------------------

@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("M", [128, 256])
def test_identity_B_reproduces_A(fused, M):
    """B = I (K = N): C must equal A times its scales exactly; any mix-up of
    rows, K order, swizzle or scale-factor placement shows up here.  M = 256
    runs the CTA-pair kernel (two 128-row halves, B split across the pair)."""
    R, ka = 2, 128
    K = N = R * ka
    w = inputs.Workload("identity", R, M, ka, N, 64, 2, 0)
    A = inputs.random_codes((M, K), 101)
    sA = inputs.random_scales((M, K // 32), 102, 117, 137)
    B = torch.zeros((N, K), dtype=torch.uint8)
    B[torch.arange(N), torch.arange(K)] = 0x38
    sB = torch.full((N, K // 32), 127, dtype=torch.uint8)
    x = {"A_seg": [A[:, r * ka:(r + 1) * ka].contiguous() for r in range(R)],
         "A_scale_seg": [sA[:, r * ka // 32:(r + 1) * ka // 32].contiguous() for r in range(R)],
         "B": B, "B_scale": sB}
    d = gu.to_device(x)
    with _plan(w) as p:
        C = gu.run_gpu(p, d, M, N, fused=fused)
        torch.cuda.synchronize()
        _status_ok(p)
        got = gu.host_bits(C)
    ref = gu.oracle_full(x)
    gv, rv = gu.bits_to_f64(got), gu.bits_to_f64(ref)
    assert np.array_equal(gv, rv), f"{np.sum(gv != rv)} of {gv.size} differ"


ELEM_PAIRS = [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")]


def _finite(codes: torch.Tensor, fmt: str) -> torch.Tensor:
    """Replace NaN / infinity codes of a format with small finite ones."""
    c = codes.clone()
    if fmt == "e5m2":
        bad = ((c >> 2) & 0x1F) == 31
        c[bad] = c[bad] & 0x83
    else:
        bad = (c & 0x7F) == 0x7F
        c[bad] = c[bad] & 0xF8
    return c


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("a_fmt,b_fmt", [("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e5m2", "e5m2")])
def test_identity_B_other_element_formats(a_fmt, b_fmt, fused):
    """The element-type fields of the MMA: with B = I in its own format
    (1.0 = 0x3C in E5M2, 0x38 in E4M3) C equals A, read in A's format, exactly."""
    R, ka, M = 2, 128, 128
    K = N = R * ka
    w = inputs.Workload("identity_fmt", R, M, ka, N, 64, 2, 0, a_fmt=a_fmt, b_fmt=b_fmt)
    A = _finite(inputs.random_codes((M, K), 111), a_fmt)
    sA = inputs.random_scales((M, K // 32), 112, 117, 137)
    B = torch.zeros((N, K), dtype=torch.uint8)
    B[torch.arange(N), torch.arange(K)] = 0x3C if b_fmt == "e5m2" else 0x38
    sB = torch.full((N, K // 32), 127, dtype=torch.uint8)
    x = {"A_seg": [A[:, r * ka:(r + 1) * ka].contiguous() for r in range(R)],
         "A_scale_seg": [sA[:, r * ka // 32:(r + 1) * ka // 32].contiguous() for r in range(R)],
         "B": B, "B_scale": sB, "workload": w}
    d = gu.to_device(x)
    with _plan(w, elem_types=mxa2a.ELEM_TYPES[(a_fmt, b_fmt)]) as p:
        C = gu.run_gpu(p, d, M, N, fused=fused)
        torch.cuda.synchronize()
        _status_ok(p)
        got = gu.host_bits(C)
    ref = gu.oracle_full(x)
    gv, rv = gu.bits_to_f64(got), gu.bits_to_f64(ref)
    assert np.array_equal(gv, rv), f"{np.sum(gv != rv)} of {gv.size} differ"


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("a_fmt,b_fmt", ELEM_PAIRS)
def test_other_element_formats_against_oracle(a_fmt, b_fmt, fused):
    """Quantised N(0,1) inputs in the other element formats, several tiles and
    a ragged N tail, against the oracle element by element."""
    w = inputs.Workload("fmt", 3, 384, 256, 528, 128, 2, 97, a_fmt=a_fmt, b_fmt=b_fmt)
    _check_full(w, fused=fused, elem_types=mxa2a.ELEM_TYPES[(a_fmt, b_fmt)])


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("a_fmt,b_fmt", ELEM_PAIRS)
def test_other_element_formats_cta_pair(a_fmt, b_fmt, fused):
    """The same on the CTA-pair kernel (its idesc takes the element types too;
    the fused path's default on large problems), against the oracle."""
    w = inputs.Workload("fmtpair", 3, 512, 256, 528, 128, 4, 99, a_fmt=a_fmt, b_fmt=b_fmt)
    with _plan(w, cta_pair=1) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR if fused else mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED) == 1
    _check_full(w, fused=fused, cta_pair=1, elem_types=mxa2a.ELEM_TYPES[(a_fmt, b_fmt)])


@pytest.mark.parametrize("M", [128, 256])
def test_scale_factors_per_block_and_column(M):
    """One-hot B with varied B scales per 32-block and column: exercises every
    scale-factor lane/column/byte position of both operands."""
    R, ka, N = 2, 256, 256
    K = R * ka
    w = inputs.Workload("onehot", R, M, ka, N, 128, 2, 0)
    rng = np.random.default_rng(7)
    perm = rng.integers(0, K, size=N)
    A = inputs.random_codes((M, K), 201)
    sA = inputs.random_scales((M, K // 32), 202, 112, 142)
    B = torch.zeros((N, K), dtype=torch.uint8)
    B[torch.arange(N), torch.from_numpy(perm)] = 0x38
    sB = inputs.random_scales((N, K // 32), 203, 120, 134)
    x = {"A_seg": [A[:, r * ka:(r + 1) * ka].contiguous() for r in range(R)],
         "A_scale_seg": [sA[:, r * ka // 32:(r + 1) * ka // 32].contiguous() for r in range(R)],
         "B": B, "B_scale": sB}
    d = gu.to_device(x)
    with _plan(w) as p:
        C = gu.run_gpu(p, d, M, N)
        torch.cuda.synchronize()
        _status_ok(p)
        got = gu.host_bits(C)
    ref = gu.oracle_full(x)
    assert np.array_equal(gu.bits_to_f64(got), gu.bits_to_f64(ref))


@pytest.mark.parametrize("fused", [True, False])
def test_e8m0_range_ends(fused):
    """Scale bytes at both ends of the E8M0 range (254 = 2^127, 1 = 2^-126) in
    the first 32-wide K block of some A rows and some B columns, all codes of
    that block positive (so no infinities of both signs meet in one sum): the
    products of two high scales overflow fp32 inside the tensor core (+inf),
    two low scales underflow to zero, a high and a low scale give ordinary
    values.  Compared with the oracle per element (matching infinities are
    equal)."""
    R, ka, M, N = 2, 128, 256, 256
    K = R * ka
    w = inputs.Workload("e8m0_ends", R, M, ka, N, 128, 2, 0)
    x = inputs.make_inputs(inputs.Workload("e8m0_src", R, M, ka, N, 128, 2, 61))
    A = torch.cat(x["A_seg"], dim=1).clone()
    sA = torch.cat(x["A_scale_seg"], dim=1).clone()
    B, sB = x["B"].clone(), x["B_scale"].clone()
    A[:, :32] &= 0x7F                     # block 0 of every row and column: positive codes
    B[:, :32] &= 0x7F
    sA[0:64, 0] = 254
    sA[64:128, 0] = 1
    sA[128:160, 0] = 253
    sB[0:64, 0] = 254
    sB[64:128, 0] = 1
    sB[128:160, 0] = 2
    x = {"A_seg": [A[:, r * ka:(r + 1) * ka].contiguous() for r in range(R)],
         "A_scale_seg": [sA[:, r * ka // 32:(r + 1) * ka // 32].contiguous() for r in range(R)],
         "B": B.contiguous(), "B_scale": sB.contiguous()}
    d = gu.to_device(x)
    with _plan(w, split_k=1) as p:
        C = gu.run_gpu(p, d, M, N, fused=fused)
        torch.cuda.synchronize()
        _status_ok(p)
        got = gu.host_bits(C)
    ref = gu.oracle_full(x)
    st = gu.assert_parity(got, ref, f"e8m0 range ends fused={fused}")
    assert st["inf_matched"] > 0      # the high x high cells did overflow on both sides


# --- the smallest workload, and small shapes spanning tiles with ragged tails -------------

@pytest.mark.parametrize("fused", [True, False])
def test_workload_tiny(fused):
    _check_full(inputs.workload(0), fused=fused)


SMALL = [
    # name, R, M, ka, N, cm, bn
    ("tiles_ragged_n", 3, 384, 256, 528, 128, 2),
    ("cm64_tail_tile", 2, 192, 128, 256, 64, 2),
    ("cm192_straddle", 2, 384, 128, 272, 192, 2),
    ("many_steps_bn2", 2, 1024, 128, 256, 64, 2),
    ("single_slot", 2, 512, 128, 256, 128, 1),
    ("bn3", 2, 768, 128, 256, 128, 3),
    ("one_segment", 1, 256, 512, 256, 128, 2),
    ("n16", 2, 128, 128, 16, 64, 2),
    ("one_step", 4, 256, 128, 512, 256, 2),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes(case):
    name, R, M, ka, N, cm, bn = case
    w = inputs.Workload(name, R, M, ka, N, cm, bn, 11)
    _check_full(w, fused=True)
    _check_full(w, fused=False)
    # with the same K split both paths issue the same MMAs in the same order
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=1) as p:
        got_f = gu.host_bits(gu.run_gpu(p, d, M, N, fused=True))
        got_u = gu.host_bits(gu.run_gpu(p, d, M, N, fused=False))
    assert np.array_equal(got_f, got_u), "fused and unfused differ"


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_narrow_tiles_match_wide(case):
    """The 128-column tile (two TMEM accumulators, items alternating between
    them) against the oracle and, bit for bit, against the 256-column tile: an
    output element sees the same MMAs in the same K order either way."""
    name, R, M, ka, N, cm, bn = case
    w = inputs.Workload(name, R, M, ka, N, cm, bn, 11)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    ref = gu.oracle_full(x)
    outs = {}
    for tile in (128, 256):
        # grid 2: each CTA runs several items, so both accumulators are reused
        with _plan(w, tile_n=tile, split_k=1, grid=2, tail_split=0) as p:
            assert p.get_option(mxa2a.MXA2A_INFO_TILE_N_FUSED) == tile
            assert p.get_option(mxa2a.MXA2A_INFO_TILE_N_UNFUSED) == tile
            for fused in (True, False):
                outs[(tile, fused)] = gu.host_bits(gu.run_gpu(p, d, M, N, fused=fused))
                torch.cuda.synchronize()
                _status_ok(p)
    gu.assert_parity(outs[(128, True)], ref, f"{name} narrow fused")
    gu.assert_parity(outs[(128, False)], ref, f"{name} narrow unfused")
    for fused in (True, False):
        assert np.array_equal(outs[(128, fused)], outs[(256, fused)]), f"narrow != wide, fused={fused}"


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_direct_read_matches_unfused(case):
    """The direct-read variant (A read in place from the segments) against the
    oracle and, bit for bit, against the unfused path at the same K split."""
    name, R, M, ka, N, cm, bn = case
    w = inputs.Workload(name, R, M, ka, N, cm, bn, 11)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=1) as p:
        got_d = gu.host_bits(gu.run_gpu(p, d, M, N, fused="direct"))
        got_u = gu.host_bits(gu.run_gpu(p, d, M, N, fused=False))
        torch.cuda.synchronize()
        _status_ok(p)
    gu.assert_parity(got_d, gu.oracle_full(x), f"{name} direct")
    assert np.array_equal(got_d, got_u), "direct and unfused differ"


def test_direct_read_split_and_new_segment_pointers():
    """Split K, and a second run with other segment buffers (the tensor maps
    are re-encoded)."""
    w = inputs.Workload("direct_split", 4, 256, 256, 512, 128, 2, 73)
    x1 = inputs.make_inputs(w)
    x2 = inputs.make_inputs(inputs.Workload("direct_split", 4, 256, 256, 512, 128, 2, 74))
    with _plan(w, split_k=2) as p:
        for x in (x1, x2, x1):
            d = gu.to_device(x)
            got = gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused="direct"))
            torch.cuda.synchronize()
            _status_ok(p)
            gu.assert_parity(got, gu.oracle_full(x), "direct split")


@pytest.mark.parametrize("split", [1, 2])
def test_step_credits_and_copy_skew_same_bits(split):
    """The whole-step staging protocol (a slot refilled only after every reader
    finished the whole previous step; readers wait for the whole step) and the
    per-segment credits, each with and without slowed copies on every 4th CTA:
    the oracle's results and, bit for bit, one another.  8 steps through a
    2-slot ring, so every slot is reused three times."""
    w = inputs.Workload("stepcred", 4, 1024, 256, 768, 128, 2, 83)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    outs = {}
    for sc in (0, 1):
        for skew in (0, 20_000):
            with _plan(w, split_k=split, grid=8, step_credits=sc, copy_skew_ns=skew) as p:
                assert p.get_option(mxa2a.MXA2A_OPT_STEP_CREDITS) == sc
                assert p.get_option(mxa2a.MXA2A_OPT_COPY_SKEW_NS) == skew
                outs[(sc, skew)] = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
                torch.cuda.synchronize()
                _status_ok(p)
    gu.assert_parity(outs[(1, 20_000)], gu.oracle_full(x), "whole-step credits with skew")
    for k, v in outs.items():
        assert np.array_equal(v, outs[(0, 0)]), f"step_credits, skew = {k} differs"


@pytest.mark.parametrize("group", [0, 1, 2, 3, 4, 8, 16])
def test_fused_raster_groups_same_bits(group):
    """Fused raster groups (n-tile outer over whole staging steps within the
    ring) against the unfused path: the same bits, and the planner's rounding
    of the requested group (0: the default, half the ring's steps)."""
    w = inputs.Workload("fgroup", 4, 2048, 256, 1040, 256, 4, 91)   # 2 m-tiles per step, 8 in the ring
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=1) as p:
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused=False))
        p.set_option(mxa2a.MXA2A_OPT_GROUP_FUSED, group)
        want = {0: 4, 1: 1, 2: 2, 3: 2, 4: 4, 8: 8, 16: 8}[group]
        assert p.get_option(mxa2a.MXA2A_INFO_GROUP_FUSED) == want
        got = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        torch.cuda.synchronize()
        _status_ok(p)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("group", [0, 1, 2, 4, 8, 16])
def test_fused_raster_groups_cta_pair(group):
    """The same with the CTA-pair kernel, whose groups count pairs of m-tiles
    (one per staging step here, 4 in the ring; the request in m-tiles halved)."""
    w = inputs.Workload("fgrouppair", 4, 2048, 256, 1040, 256, 4, 93)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=1, cta_pair=1) as p:
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused=False))
        p.set_option(mxa2a.MXA2A_OPT_GROUP_FUSED, group)
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR) == 1
        want = {0: 2, 1: 1, 2: 1, 4: 2, 8: 4, 16: 4}[group]
        assert p.get_option(mxa2a.MXA2A_INFO_GROUP_FUSED) == want
        got = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        torch.cuda.synchronize()
        _status_ok(p)
    assert np.array_equal(got, ref)


def test_step_credit_options_validated():
    w = inputs.workload(0)
    with _plan(w) as p:
        assert p.get_option(mxa2a.MXA2A_OPT_STEP_CREDITS) == 0
        for key, bad in ((mxa2a.MXA2A_OPT_STEP_CREDITS, 2), (mxa2a.MXA2A_OPT_COPY_SKEW_NS, -1),
                         (mxa2a.MXA2A_OPT_COPY_SKEW_NS, 2_000_000)):
            with pytest.raises(mxa2a.Mxa2aError):
                p.set_option(key, bad)


@pytest.mark.parametrize("split", [2, 3])
def test_narrow_tiles_split_k(split):
    w = inputs.Workload("nsplit", 6, 256, 256, 640, 128, 2, 71)
    got_f, _ = _check_full(w, fused=True, split_k=split, tile_n=128)
    got_u, _ = _check_full(w, fused=False, split_k=split, tile_n=128)
    assert np.array_equal(got_f, got_u)


@pytest.mark.parametrize("split", [2, 3, 6])
def test_forced_split_k(split):
    w = inputs.Workload("split", 6, 256, 256, 512, 128, 2, 13)
    got_f, _ = _check_full(w, fused=True, split_k=split)
    got_u, _ = _check_full(w, fused=False, split_k=split)
    assert np.array_equal(got_f, got_u)


@pytest.mark.parametrize("fused", [True, False])
def test_split_k_tiles_straddling_grid_rounds(fused):
    """K split 3 on a grid of 4 CTAs (27 items): the 3 splits of most tiles are
    run by CTAs in two consecutive rounds of the persistent grid, and each split
    waits for its siblings before it sums its share of the tile."""
    w = inputs.Workload("straddle", 6, 384, 256, 640, 128, 2, 61)
    with _plan(w, split_k=3, grid=4) as p:
        key = mxa2a.MXA2A_INFO_GRID_FUSED if fused else mxa2a.MXA2A_INFO_GRID_UNFUSED
        assert p.get_option(key) == 4
    _check_full(w, fused=fused, split_k=3, grid=4)


@pytest.mark.parametrize("fused", [True, False])
def test_tail_split_last_round(fused):
    """8 tiles (K = 8192) on a grid of 6 CTAs: the second round would hold 2
    whole tiles, so the planner splits those two along K (each half reading 1
    of the 2 segments) and 4 CTAs share them.  The tail's tiles are ragged (64
    of their rows past M, one of them with columns past N), checked against
    the oracle, against the same plan with whole tiles, and for identical bits
    over repeated runs; nothing is written past M x N."""
    w = inputs.Workload("tail", 2, 448, 4096, 400, 64, 4, 67)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    ref = gu.oracle_full(x)
    info = mxa2a.MXA2A_INFO_TAIL_SPLIT if fused else mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED
    got = {}
    for tail in (1, 0):
        with _plan(w, grid=6, tail_split=tail, split_k=1) as p:
            assert p.get_option(mxa2a.MXA2A_OPT_TAIL_SPLIT) == tail
            assert p.get_option(info) == (2 if tail else 1)
            if fused:
                assert p.get_option(mxa2a.MXA2A_INFO_ITEMS) == (6 + 2 * 2 if tail else 8)
            fn = p.run if fused else p.run_unfused
            bufs = []
            for _ in range(3):
                buf = torch.full((w.M * w.N + 4096,), -1, dtype=torch.int16, device="cuda")
                fn(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], buf[: w.M * w.N].view(w.M, w.N))
                bufs.append(buf)
            torch.cuda.synchronize()
            _status_ok(p)
        for buf in bufs:
            assert bool((buf[w.M * w.N:] == -1).all())
        bits = [gu.host_bits(b[: w.M * w.N].view(w.M, w.N)) for b in bufs]
        for b in bits[1:]:
            assert np.array_equal(bits[0], b)
        got[tail] = bits[0]
        gu.assert_parity(got[tail], ref, f"tail split {tail} fused={fused}")


def test_split_k_deterministic_over_runs():
    """The split partials are summed in a fixed order whichever split finishes
    last, so repeated runs give identical bits."""
    w = inputs.Workload("splitdet", 4, 128, 512, 2048, 128, 2, 47)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=4) as p:
        outs = [gu.host_bits(gu.run_gpu(p, d, w.M, w.N)) for _ in range(4)]
        torch.cuda.synchronize()
        _status_ok(p)
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)
    gu.assert_parity(outs[0], gu.oracle_full(x), "split 4 deterministic")


def test_automatic_split_small_m():
    w = inputs.Workload("autosplit", 8, 64, 256, 1024, 64, 2, 17, outliers=True)
    with _plan(w) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_SPLITS) > 1
    _check_full(w, fused=True)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("split,tail", [(2, 0), (1, 1)])
def test_cta_pair_split_items(fused, split, tail):
    """The CTA-pair kernel's split items, each CTA of a pair writing and
    summing its own m-tile's partials: a uniform split in two (8 items on 3
    pairs), and the tail split (4 pair tiles on 3 pairs: the fourth split in
    two, a slot per CTA); against the oracle, identical bits over runs."""
    w = inputs.Workload("pairsplit", 2, 512, 4096, 400, 64, 4, 73)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, cta_pair=1, split_k=split, grid=6, tail_split=tail) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR if fused else mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED) == 1
        assert p.get_option(mxa2a.MXA2A_INFO_SPLITS if fused else mxa2a.MXA2A_INFO_SPLITS_UNFUSED) == split
        assert p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT if fused else mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED) == \
            (2 if tail else 1)
        outs = [gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused=fused)) for _ in range(2)]
        torch.cuda.synchronize()
        _status_ok(p)
    assert np.array_equal(outs[0], outs[1])
    gu.assert_parity(outs[0], gu.oracle_full(x), f"pair split={split} tail={tail} fused={fused}")


@pytest.mark.parametrize("fused", [True, False])
def test_cta_pair_kernel_against_single_cta_kernel(fused):
    """The CTA-pair kernel (256-row tiles, .cta_group::2 MMAs issued by the even
    CTA) and the single-CTA kernel agree with the oracle and with each other."""
    w = inputs.Workload("pair", 3, 768, 256, 1040, 128, 2, 59)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    outs = {}
    for pair in (1, 0):
        with _plan(w, cta_pair=pair, split_k=1) as p:
            assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR if fused else mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED) == pair
            C = gu.run_gpu(p, d, w.M, w.N, fused=fused)
            torch.cuda.synchronize()
            _status_ok(p)
            outs[pair] = gu.host_bits(C)
    ref = gu.oracle_full(x)
    gu.assert_parity(outs[1], ref, f"pair fused={fused}")
    gu.assert_parity(outs[0], ref, f"single fused={fused}")
    diff = gu.parity_stats(outs[1], outs[0])
    assert diff["fail"] == 0, diff


def test_zigzag_rotation_off_same_tolerance():
    w = inputs.Workload("noswizzle", 4, 512, 256, 768, 128, 2, 19)
    _check_full(w, fused=True, zigzag=0, rotate=0)


def test_unfused_raster_groups_same_bits():
    """The raster group only reorders the work items: group sizes 1, 3 (a
    ragged last group over 7 m-tiles) and 16 give identical bits."""
    w = inputs.Workload("groups", 2, 896, 256, 1536, 128, 2, 61)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    outs = []
    for g in (1, 3, 16):
        with _plan(w, group_m=g, split_k=1, grid=5) as p:
            assert p.get_option(mxa2a.MXA2A_INFO_GROUP_UNFUSED) == min(g, 7)
            outs.append(gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused=False)))
            torch.cuda.synchronize()
            _status_ok(p)
    gu.assert_parity(outs[0], gu.oracle_full(x), "raster group 1")
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("pair", [0, 1])
def test_cuda_graph_replay_matches_eager(fused, pair):
    """A run captured into a CUDA graph and replayed gives the eager run's bits
    (the flags, and the CTA-pair kernel's inline B-scale pack count, reset
    themselves at the end of every launch)."""
    w = inputs.Workload("graph", 2, 256, 256, 512, 128, 2, 83)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=1, cta_pair=pair) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR if fused else mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED) == pair
        eager = gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused=fused))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        C = torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda")
        fn = p.run if fused else p.run_unfused
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C, side)
        for _ in range(3):
            C.fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(gu.host_bits(C), eager)
        _status_ok(p)
    gu.assert_parity(eager, gu.oracle_full(x), f"graph fused={fused} pair={pair}")


def test_cuda_graph_capture_leaves_the_tail_whole():
    """A plan with a tail split can be captured: the captured run takes its
    last round's tiles whole (split partials are tagged with the launch index,
    which a replay repeats), so every replay gives the bits of an eager run
    without the tail split."""
    w = inputs.Workload("graphtail", 2, 448, 4096, 400, 64, 4, 71)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, grid=6, tail_split=0, split_k=1) as p:
        whole = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        torch.cuda.synchronize()
    with _plan(w, grid=6, split_k=1) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT) == 2
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        C = torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            p.run(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C, side)
        for _ in range(3):
            C.fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(gu.host_bits(C), whole)
        _status_ok(p)
    gu.assert_parity(whole, gu.oracle_full(x), "graph tail")


def test_cuda_graph_capture_refuses_split():
    w = inputs.Workload("graphsplit", 4, 128, 256, 256, 64, 2, 89)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=2) as p:
        gu.run_gpu(p, d, w.M, w.N)   # eager runs are fine
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        C = torch.empty((w.M, w.N), dtype=torch.int16, device="cuda")
        g = torch.cuda.CUDAGraph()
        with pytest.raises(mxa2a.Mxa2aError) as e:
            with torch.cuda.graph(g, stream=side):
                p.run(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C, side)
        assert e.value.code == mxa2a.MXA2A_ERR_CAPTURE_SPLIT


def test_small_grid_many_items_per_cta():
    w = inputs.Workload("grid3", 3, 512, 128, 768, 64, 2, 23)
    _check_full(w, fused=True, grid=3)


def test_repeat_runs_identical_and_counters_reset():
    w = inputs.Workload("repeat", 2, 512, 128, 512, 64, 2, 29)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w) as p:
        outs = [gu.host_bits(gu.run_gpu(p, d, w.M, w.N)) for _ in range(3)]
        torch.cuda.synchronize()
        _status_ok(p)
        flags = p.read_workspace(mxa2a.MXA2A_WS_FLAGS).view(np.uint64)
        assert np.all(flags == 0)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_non_default_stream_and_host_entry():
    w = inputs.workload(0)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    s = torch.cuda.Stream()
    with _plan(w) as p:
        C = gu.run_gpu(p, d, w.M, w.N, stream=s)
        s.synchronize()
        got = gu.host_bits(C)
        hA = [a.pin_memory() for a in x["A_seg"]]
        hS = [a.pin_memory() for a in x["A_scale_seg"]]
        hB, hBs = x["B"].pin_memory(), x["B_scale"].pin_memory()
        hC = torch.empty((w.M, w.N), dtype=torch.int16).pin_memory()
        p.run_host(hA, hS, hB, hBs, hC, s)
        s.synchronize()
        _status_ok(p)
    assert np.array_equal(got, hC.numpy().view(np.uint16))
    gu.assert_parity(got, gu.oracle_full(x), "stream")


def test_host_entry_pinned_and_pageable_same_bits():
    """mxa2a_run_host with pinned host buffers (inputs read or copied by the SMs,
    a pinned C written by the epilogue itself) and with pageable ones (DMA
    copies), and a mix: the same bits as the device entry.  N = 400 leaves a
    ragged 16-column tail in the last 32-column chunk."""
    w = inputs.Workload("hostcopy", 3, 384, 256, 400, 128, 2, 97)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w) as p:
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        outs = []
        for pin_in, pin_out in ((True, True), (False, False), (True, False), (False, True)):
            cv = (lambda t: t.pin_memory()) if pin_in else (lambda t: t.clone())
            hA = [cv(a) for a in x["A_seg"]]
            hS = [cv(s) for s in x["A_scale_seg"]]
            hC = torch.full((w.M, w.N), -1, dtype=torch.int16)
            if pin_out:
                hC = hC.pin_memory()
            p.run_host(hA, hS, cv(x["B"]), cv(x["B_scale"]), hC)
            torch.cuda.synchronize()
            _status_ok(p)
            outs.append(hC.numpy().view(np.uint16).copy())
    for o in outs:
        assert np.array_equal(o, ref)


def test_host_entry_pinned_output_with_split_k():
    """The split-K sums also write a pinned C through its device view."""
    w = inputs.Workload("hostsplit", 4, 256, 256, 528, 128, 2, 101)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=3) as p:
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        hA = [a.pin_memory() for a in x["A_seg"]]
        hS = [a.pin_memory() for a in x["A_scale_seg"]]
        hC = torch.full((w.M, w.N), -1, dtype=torch.int16).pin_memory()
        p.run_host(hA, hS, x["B"].pin_memory(), x["B_scale"].pin_memory(), hC)
        torch.cuda.synchronize()
        _status_ok(p)
    assert np.array_equal(hC.numpy().view(np.uint16), ref)
    gu.assert_parity(ref, gu.oracle_full(x), "hostsplit")


@pytest.mark.parametrize("tail", [0, 1])
def test_host_entry_pinned_output_cta_pair(tail):
    """The CTA-pair kernel's epilogue writes a pinned C through its device view
    (each CTA of a pair its own rows; with the tail split, the sums too): the
    device run's bits, nothing past M x N."""
    w = inputs.Workload("hostpair", 2, 512, 4096, 400, 64, 4, 109)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, cta_pair=1, grid=6, split_k=1, tail_split=tail) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR) == 1
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        hA = [a.pin_memory() for a in x["A_seg"]]
        hS = [a.pin_memory() for a in x["A_scale_seg"]]
        guard = torch.full((w.M + 1, w.N), -1, dtype=torch.int16).pin_memory()
        p.run_host(hA, hS, x["B"].pin_memory(), x["B_scale"].pin_memory(), guard[: w.M])
        torch.cuda.synchronize()
        _status_ok(p)
    assert np.array_equal(guard[: w.M].numpy().view(np.uint16), ref)
    assert bool((guard[w.M] == -1).all())
    gu.assert_parity(ref, gu.oracle_full(x), f"hostpair tail={tail}")


def test_host_entry_automatic_pairs_run_single_cta():
    """A plan whose fused path is automatically on CTA pairs runs a pinned-C
    host call on single CTAs (the host link bounds it) and keeps its choice:
    the device run's bits (no tail split on either kernel here)."""
    w = inputs.Workload("hostauto", 2, 512, 4096, 400, 128, 4, 111)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, grid=4, split_k=1) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR) == 1
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        hA = [a.pin_memory() for a in x["A_seg"]]
        hS = [a.pin_memory() for a in x["A_scale_seg"]]
        hC = torch.full((w.M, w.N), -1, dtype=torch.int16).pin_memory()
        p.run_host(hA, hS, x["B"].pin_memory(), x["B_scale"].pin_memory(), hC)
        torch.cuda.synchronize()
        _status_ok(p)
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR) == 1
        again = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        torch.cuda.synchronize()
    assert np.array_equal(hC.numpy().view(np.uint16), ref)
    assert np.array_equal(again, ref)
    gu.assert_parity(ref, gu.oracle_full(x), "hostauto")


def test_automatic_cta_pair_choice():
    """Automatic (default): the fused path on pairs only when the staging window
    holds at least two pair tiles per resident pair (the 8 x 8192^3 benchmark
    problem: 256), never the unfused path; the 2048-row problem's window holds
    32 and stays on single CTAs."""
    for idx, fused_pair in ((3, 1), (1, 0)):
        w = inputs.workload(idx)
        with _plan(w) as p:
            assert p.get_option(mxa2a.MXA2A_OPT_CTA_PAIR) == 2
            assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR) == fused_pair, w.name
            assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED) == 0, w.name


def test_host_entry_pinned_output_with_tail_split():
    """The tail split's sums write a pinned C through its device view: the
    same bits as the device run (whose tail is split too), nothing past M x N."""
    w = inputs.Workload("hosttail", 2, 448, 4096, 400, 64, 4, 107)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, grid=6, split_k=1) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT) == 2
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        hA = [a.pin_memory() for a in x["A_seg"]]
        hS = [a.pin_memory() for a in x["A_scale_seg"]]
        guard = torch.full((w.M + 1, w.N), -1, dtype=torch.int16).pin_memory()
        p.run_host(hA, hS, x["B"].pin_memory(), x["B_scale"].pin_memory(), guard[: w.M])
        torch.cuda.synchronize()
        _status_ok(p)
    assert np.array_equal(guard[: w.M].numpy().view(np.uint16), ref)
    assert bool((guard[w.M] == -1).all())
    gu.assert_parity(ref, gu.oracle_full(x), "hosttail")


@pytest.mark.parametrize("split", [1, 4])
def test_host_entry_pinned_output_rows_and_columns_past_the_ends(split):
    """M = 64 (half a tile) and N = 400 (a ragged last tile): the epilogue's
    stores to a pinned C skip the rows past M and the columns past N, with K
    unsplit (whole 256-byte row pieces) and split 4 (the split sums' pieces)."""
    w = inputs.Workload("hostm64", 4, 64, 256, 400, 64, 2, 103)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, split_k=split) as p:
        ref = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
        hA = [a.pin_memory() for a in x["A_seg"]]
        hS = [a.pin_memory() for a in x["A_scale_seg"]]
        # one pinned buffer with a guard row after C: nothing may be written past M x N
        guard = torch.full((w.M + 1, w.N), -1, dtype=torch.int16).pin_memory()
        p.run_host(hA, hS, x["B"].pin_memory(), x["B_scale"].pin_memory(), guard[:w.M])
        torch.cuda.synchronize()
        _status_ok(p)
    out = guard.numpy().view(np.uint16)
    assert np.array_equal(out[:w.M], ref)
    assert np.all(out[w.M] == 0xFFFF)
    gu.assert_parity(ref, gu.oracle_full(x), f"hostm64 split {split}")


def test_zero_A_gives_zero():
    w = inputs.Workload("zero", 2, 128, 128, 256, 64, 2, 0)
    x = inputs.make_inputs(w)
    x["A_seg"] = [torch.zeros_like(a) for a in x["A_seg"]]
    d = gu.to_device(x)
    with _plan(w) as p:
        got = gu.host_bits(gu.run_gpu(p, d, w.M, w.N))
    assert np.all(gu.bits_to_f64(got) == 0)


# --- building blocks: the staging exchange and the scale-factor layouts --------------------

def _atom_restate(sf: np.ndarray, rows_pad: int) -> np.ndarray:
    """CPU restatement of the MMA scale atom layout: [K/128][rows_pad/128][512]."""
    rows, kb32 = sf.shape
    kbs = kb32 // 4
    out = np.zeros((kbs, rows_pad // 128, 128, 4), dtype=np.uint8)
    for x in range(rows):
        g, xi = divmod(x, 128)
        word = (xi % 32) * 4 + xi // 32
        for kb in range(kbs):
            out[kb, g, word] = sf[x, kb * 4:(kb + 1) * 4]
    return out.reshape(-1)


def test_exchange_only_ring_and_scales():
    """Only the staging copy runs (buffer_num >= steps): the ring must hold the
    segments byte for byte at [slot][r][row], the scales in the MMA layout."""
    w = inputs.Workload("xchg", 3, 256, 256, 256, 64, 4, 31)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w, exchange_only=1) as p:
        gu.run_gpu(p, d, w.M, w.N)
        torch.cuda.synchronize()
        _status_ok(p)
        ring = p.read_workspace(mxa2a.MXA2A_WS_RING).reshape(w.buffer_num, w.R, w.commMSize, w.kPerRank)
        sfa = p.read_workspace(mxa2a.MXA2A_WS_SFA)
    for s in range(w.M // w.commMSize):
        for r in range(w.R):
            src = x["A_seg"][r].numpy()[s * w.commMSize:(s + 1) * w.commMSize]
            assert np.array_equal(ring[s % w.buffer_num, r], src), (s, r)
    sf_full = np.concatenate([s.numpy() for s in x["A_scale_seg"]], axis=1)
    assert np.array_equal(sfa, _atom_restate(sf_full, 128 * ((w.M + 127) // 128)))


def test_b_scale_pack_layout():
    w = inputs.Workload("sfb", 2, 128, 256, 400, 64, 2, 37)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w) as p:
        gu.run_gpu(p, d, w.M, w.N)
        torch.cuda.synchronize()
        sfb = p.read_workspace(mxa2a.MXA2A_WS_SFB)
    npad = 256 * ((w.N + 255) // 256)
    assert np.array_equal(sfb, _atom_restate(x["B_scale"].numpy(), npad))


def test_unfused_pack_matches_concatenation():
    w = inputs.Workload("pack", 3, 192, 128, 256, 64, 2, 41)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w) as p:
        gu.run_gpu(p, d, w.M, w.N, fused=False)
        torch.cuda.synchronize()
        ap = p.read_workspace(mxa2a.MXA2A_WS_APACKED).reshape(w.M, w.K)
    assert np.array_equal(ap, np.concatenate([a.numpy() for a in x["A_seg"]], axis=1))


# --- error handling ---------------------------------------------------------------------------

def test_create_rejects_bad_shapes():
    with pytest.raises(mxa2a.Mxa2aError) as e:
        mxa2a.Plan(2, 0, 128, 256, 64, 2)
    assert e.value.code == mxa2a.MXA2A_ERR_INVALID_SHAPE
    with pytest.raises(mxa2a.Mxa2aError) as e:
        mxa2a.Plan(2, 100, 128, 256, 64, 2)
    assert e.value.code == mxa2a.MXA2A_ERR_INVALID_SHAPE


def test_run_rejects_misaligned_pointers():
    w = inputs.workload(0)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w) as p:
        C = torch.empty((w.M * w.N + 8,), dtype=torch.int16, device="cuda")
        with pytest.raises(mxa2a.Mxa2aError) as e:
            p.run(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C.data_ptr() + 2)
        assert e.value.code == mxa2a.MXA2A_ERR_MISALIGNED


# --- full-size workloads: sampled rows, all columns ---------------------------------------

@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_workloads_sampled(idx):
    w = inputs.workload(idx)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    rows = gu.sample_rows(w.M, 40 if w.M > 64 else w.M, seed=idx)
    if w.M >= 1024:
        # the last m-tiles hold the tiles of the grid's last round (split in K on both paths)
        rows = np.unique(np.concatenate([rows, [w.M - 700, w.M - 200, w.M - 65, w.M - 1]]))
    with _plan(w, timeout_ns=2_000_000_000) as p:
        Cf = gu.run_gpu(p, d, w.M, w.N, fused=True)
        Cu = gu.run_gpu(p, d, w.M, w.N, fused=False)
        torch.cuda.synchronize()
        _status_ok(p)
        got_f = gu.host_bits(Cf)
        got_u = gu.host_bits(Cu)
        same_split = p.get_option(mxa2a.MXA2A_INFO_SPLITS) == p.get_option(mxa2a.MXA2A_INFO_SPLITS_UNFUSED)
        whole_f, whole_u = got_f, got_u
        if (p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT), p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED)) != (1, 1):
            # the paths' last rounds hold different tiles (their raster orders differ):
            # compare the two paths bit for bit with whole tiles
            p.set_option(mxa2a.MXA2A_OPT_TAIL_SPLIT, 0)
            whole_f = gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused=True))
            whole_u = gu.host_bits(gu.run_gpu(p, d, w.M, w.N, fused=False))
            torch.cuda.synchronize()
            _status_ok(p)
    ref = oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"], rows=rows)
    gu.assert_parity(got_f[rows], ref, f"{w.name} fused sampled {len(rows)} rows")
    gu.assert_parity(got_u[rows], ref, f"{w.name} unfused sampled {len(rows)} rows")
    if whole_f is not got_f:
        gu.assert_parity(whole_f[rows], ref, f"{w.name} fused, whole tiles, sampled {len(rows)} rows")
    if same_split:
        assert np.array_equal(whole_f, whole_u), "fused and unfused differ"
    # every output written (no NaN left from the 0xFFFF fill), magnitudes sane
    assert not np.isnan(gu.bits_to_f64(got_f)).any()


def _random_shapes(n, seed):
    """Seeded legal shapes: R 1..6, kPerRank 128..512, commMSize 64..256 in
    steps of 64, M 1..8 staging steps, N 16..592 in steps of 16, buffer_num
    1..4 and at least the staging steps one 128-row tile spans (2 when
    commMSize is not a multiple of 128).  The rules are restated here so the
    shapes exist before the library is loaded."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        R = int(rng.integers(1, 7))
        ka = 128 * int(rng.integers(1, 5))
        cm = 64 * int(rng.integers(1, 5))
        M = cm * int(rng.integers(1, 9))
        N = 16 * int(rng.integers(1, 38))
        bn = int(rng.integers(1, 5))
        if bn < (1 if cm % 128 == 0 else 2):
            continue
        out.append((R, M, ka, N, cm, bn, int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("shape", _random_shapes(16, 2026), ids=lambda s: "r{}_m{}_ka{}_n{}_cm{}_bn{}".format(*s[:6]))
def test_random_shapes_all_paths(shape):
    """A seeded sweep of legal shapes: fused, unfused and direct against the
    oracle, and bitwise equal to each other at the same K split."""
    R, M, ka, N, cm, bn, seed = shape
    assert mxa2a.mxa2a_validate(R, M, ka, N, cm, bn) == mxa2a.MXA2A_OK
    w = inputs.Workload("sweep", R, M, ka, N, cm, bn, seed)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with _plan(w) as p:
        p.set_option(mxa2a.MXA2A_OPT_SPLIT_K, p.get_option(mxa2a.MXA2A_INFO_SPLITS))   # one split for all paths
        got = {f: gu.host_bits(gu.run_gpu(p, d, M, N, fused=f)) for f in (True, False, "direct")}
        torch.cuda.synchronize()
        _status_ok(p)
    gu.assert_parity(got[True], gu.oracle_full(x), f"sweep {shape}")
    assert np.array_equal(got[True], got[False]) and np.array_equal(got[True], got["direct"])
