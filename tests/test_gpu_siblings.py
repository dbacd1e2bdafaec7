"""GPU parity of the sibling fused operators through the C ABI: AllGather +
GEMM, GEMM + ReduceScatter and GEMM + AllReduce (one-shot) (the performance
optimisation guide, sections 3.1 to 3.3) against the CPU oracle.

Gates.  AllGather + GEMM, and the blocks GEMM + ReduceScatter sends, are GEMM
outputs: per element |gpu - ref| <= 1e-2 + 1e-2*|ref|, as for the all-to-all.
The reduced output (of the reduce-scatter and of the all-reduce) adds one
term: this rank's partial is rounded to BF16
before the sum (the operation's definition), and where the fp32 accumulation
lands on the other side of a BF16 rounding midpoint than the exact product,
the rounded partial differs by one BF16 spacing of |P| (2^(floor(log2|P|)-7)),
which the sum carries.  So the output's gate is 1e-2 + 1e-2*|ref| + that
spacing of the exact partial.  Fused and unfused runs give the same bits.
"""
from __future__ import annotations

import dataclasses

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


def _status_ok(p):
    st = p.status()
    assert st["code"] == 0, st


# --- AllGather + GEMM ----------------------------------------------------------------

def _ag_plan(w, **opts):
    p = mxa2a.AllGatherPlan(w.R, w.rowsPerRank, w.K, w.N, w.commMSize, w.buffer_num)
    p.set_option(mxa2a.MXA2A_OPT_TIMEOUT_NS, 500_000_000)
    for k, v in opts.items():
        p.set_option(getattr(mxa2a, "MXA2A_OPT_" + k.upper()), v)
    return p


def _ag_dev(x):
    return ([a.cuda() for a in x["A_blk"]], [s.cuda() for s in x["A_scale_blk"]], x["B"].cuda(),
            x["B_scale"].cuda())


def _ag_run(p, dev, M, N, path):
    A, S, B, Bs = dev
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    {"fused": p.run, "unfused": p.run_unfused, "direct": p.run_direct}[path](A, S, B, Bs, C)
    torch.cuda.synchronize()
    _status_ok(p)
    return gu.host_bits(C)


AG_SMALL = [
    inputs.AG_WORKLOADS[0],                                                        # 3 x 128 rows, 64-row steps
    inputs.AllGatherWorkload("ag_r2_m512_k256_n512", 2, 256, 256, 512, 128, 2, 22),
    inputs.AllGatherWorkload("ag_r5_m320_k128_n64", 5, 64, 128, 64, 64, 2, 23),   # blocks of half a tile
    inputs.AllGatherWorkload("ag_r1_m256_k512_n160", 1, 256, 512, 160, 256, 1, 24),
]


@pytest.mark.parametrize("w", AG_SMALL, ids=[w.name for w in AG_SMALL])
def test_allgather_against_oracle_and_paths_agree(w):
    x = inputs.make_allgather_inputs(w)
    dev = _ag_dev(x)
    ref = oracle.gemm_allgather(x["A_blk"], x["A_scale_blk"], x["B"], x["B_scale"])
    with _ag_plan(w) as p:
        assert p.get_option(mxa2a.MXA2A_INFO_KIND) == mxa2a.MXA2A_KIND_ALLGATHER
        assert p.get_option(mxa2a.MXA2A_INFO_SPLITS) == 1
        got = {path: _ag_run(p, dev, w.M, w.N, path) for path in ("fused", "unfused")}
        if w.rowsPerRank % 128 == 0:
            got["direct"] = _ag_run(p, dev, w.M, w.N, "direct")
        else:
            with pytest.raises(mxa2a.Mxa2aError) as e:
                _ag_run(p, dev, w.M, w.N, "direct")
            assert e.value.code == mxa2a.MXA2A_ERR_INVALID_OPTION
    gu.assert_parity(got["fused"], ref, f"{w.name} fused")
    for path, bits in got.items():
        assert np.array_equal(bits, got["fused"]), f"{path} differs from fused"


def test_allgather_full_size_sampled():
    """The benchmark's all-gather workload (4 blocks of 512 rows, K = N =
    4096) in the benchmark's launch configuration, on sampled rows."""
    w = inputs.AG_WORKLOADS[1]
    x = inputs.make_allgather_inputs(w)
    dev = _ag_dev(x)
    with _ag_plan(w) as p:
        got_f = _ag_run(p, dev, w.M, w.N, "fused")
        got_u = _ag_run(p, dev, w.M, w.N, "unfused")
        # 256 tiles on the persistent grid: the last round's tiles are split in K,
        # and the two paths' raster orders put different tiles there, so the
        # paths are compared bit for bit with whole tiles
        tails = (p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT), p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED))
        p.set_option(mxa2a.MXA2A_OPT_TAIL_SPLIT, 0)
        whole_f = _ag_run(p, dev, w.M, w.N, "fused")
        whole_u = _ag_run(p, dev, w.M, w.N, "unfused")
    rows = gu.sample_rows(w.M, 24, 3)
    rows = np.unique(np.concatenate([rows, [w.rowsPerRank - 1, w.rowsPerRank, 3 * w.rowsPerRank, w.M - 1]]))
    ref = oracle.gemm_allgather(x["A_blk"], x["A_scale_blk"], x["B"], x["B_scale"], rows=rows)
    gu.assert_parity(got_f[rows], ref, f"allgather full size, tail split {tails}")
    gu.assert_parity(got_u[rows], ref, f"allgather full size unfused, tail split {tails}")
    gu.assert_parity(whole_f[rows], ref, "allgather full size, whole tiles")
    assert np.array_equal(whole_f, whole_u)


@pytest.mark.parametrize("split,grid", [(2, 0), (1, 6)])
def test_allgather_split_items(split, grid):
    """The all-gather's split items, whose K ranges are column ranges of every
    row block: a uniform split in two (all paths the same bits), and the tail
    split (8 tiles, K = 8192, on 6 CTAs: the last 2 split in two); against the
    oracle."""
    w = inputs.AllGatherWorkload("ag_split", 2, 256, 8192, 400, 64, 4, 31)
    x = inputs.make_allgather_inputs(w)
    dev = _ag_dev(x)
    ref = oracle.gemm_allgather(x["A_blk"], x["A_scale_blk"], x["B"], x["B_scale"])
    opts = dict(split_k=split)
    if grid:
        opts["grid"] = grid
    with _ag_plan(w, **opts) as p:
        if split == 2:
            assert p.get_option(mxa2a.MXA2A_INFO_SPLITS) == 2
        else:
            assert p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT) == 2
            assert p.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED) == 2
        got = {path: _ag_run(p, dev, w.M, w.N, path) for path in ("fused", "unfused", "direct")}
    for path, bits in got.items():
        gu.assert_parity(bits, ref, f"allgather split={split} grid={grid} {path}")
    if split == 2:
        assert np.array_equal(got["fused"], got["unfused"]) and np.array_equal(got["fused"], got["direct"])


def test_allgather_host_entry_and_new_block_pointers():
    w = inputs.AG_WORKLOADS[0]
    x1 = inputs.make_allgather_inputs(w)
    x2 = inputs.make_allgather_inputs(dataclasses.replace(w, seed=99))
    with _ag_plan(w) as p:
        for x in (x1, x2):
            dev = _ag_dev(x)
            got = _ag_run(p, dev, w.M, w.N, "fused")
            assert np.array_equal(got, _ag_run(p, dev, w.M, w.N, "direct"))
            gu.assert_parity(got, oracle.gemm_allgather(x["A_blk"], x["A_scale_blk"], x["B"], x["B_scale"]),
                             "allgather new pointers")
        hA = [a.pin_memory() for a in x2["A_blk"]]
        hS = [s.pin_memory() for s in x2["A_scale_blk"]]
        hC = torch.empty((w.M, w.N), dtype=torch.int16).pin_memory()
        p.run_host(hA, hS, x2["B"].pin_memory(), x2["B_scale"].pin_memory(), hC)
        torch.cuda.synchronize()
        _status_ok(p)
    assert np.array_equal(hC.numpy().view(np.uint16), got)


# --- GEMM + ReduceScatter ------------------------------------------------------------

def _rs_dev(x):
    return (x["A"].cuda(), x["A_scale"].cuda(), x["B"].cuda(), x["B_scale"].cuda(),
            [None if r is None else r.cuda() for r in x["recv"]])


def _rs_run(p, dev, w, fused):
    A, S, B, Bs, recv = dev
    send = [None if j == w.rank else torch.full((w.rows, w.N), -1, dtype=torch.int16, device="cuda")
            for j in range(w.R)]
    out = torch.full((w.rows, w.N), -1, dtype=torch.int16, device="cuda")
    (p.run if fused else p.run_unfused)(A, S, B, Bs, recv, send, out)
    torch.cuda.synchronize()
    _status_ok(p)
    return {j: gu.host_bits(t) for j, t in enumerate(send) if t is not None}, gu.host_bits(out)


def _assert_out_parity(got, ref, P_own, label):
    g, r, pw = gu.bits_to_f64(got), gu.bits_to_f64(ref), np.abs(gu.bits_to_f64(P_own))
    _, e = np.frexp(pw)
    spacing = np.where(pw > 0, np.ldexp(1.0, e - 1 - 7), 0.0)
    tol = gu.ATOL + gu.RTOL * np.abs(r) + spacing
    bad = ~(np.abs(g - r) <= tol)
    print(f"[parity] {label} max_abs {np.abs(g - r).max():.3g} over_plain_gate "
          f"{int((np.abs(g - r) > gu.ATOL + gu.RTOL * np.abs(r)).sum())} fail {int(bad.sum())}")
    assert not bad.any(), (label, int(bad.sum()))


def _rs_check(w, dev, x):
    with mxa2a.ReduceScatterPlan(w.R, w.rank, w.M, w.K, w.N) as p:
        p.set_option(mxa2a.MXA2A_OPT_TIMEOUT_NS, 500_000_000)
        assert p.get_option(mxa2a.MXA2A_INFO_KIND) == mxa2a.MXA2A_KIND_REDUCE_SCATTER
        send_f, out_f = _rs_run(p, dev, w, True)
        send_u, out_u = _rs_run(p, dev, w, False)
    send_r, out_r = oracle.gemm_reduce_scatter(x["A"], x["A_scale"], x["B"], x["B_scale"],
                                               [None if r is None else r.numpy() for r in x["recv"]], w.R, w.rank)
    own_rows = np.arange(w.rank * w.rows, (w.rank + 1) * w.rows)
    P_own = oracle.gemm([x["A"]], [x["A_scale"]], x["B"], x["B_scale"], rows=own_rows)
    assert sorted(send_f) == sorted(send_r)
    for j in send_r:
        gu.assert_parity(send_f[j], send_r[j], f"{w.name} send[{j}]")
        assert np.array_equal(send_f[j], send_u[j]), f"send[{j}] fused != unfused"
    _assert_out_parity(out_f, out_r, P_own, f"{w.name} out")
    assert np.array_equal(out_f, out_u), "out fused != unfused"


@pytest.mark.parametrize("rank", [0, 1, 2])
def test_reduce_scatter_small_against_oracle(rank):
    w = dataclasses.replace(inputs.RS_WORKLOADS[0], rank=rank)
    x = inputs.make_reduce_scatter_inputs(w)
    _rs_check(w, _rs_dev(x), x)


@pytest.mark.parametrize("shape", [(2, 0, 128, 128, 64), (4, 3, 512, 256, 528), (1, 0, 192, 256, 256)],
                         ids=["r2_m128", "r4_m512_ntail", "r1"])
def test_reduce_scatter_shapes(shape):
    R, rank, M, K, N = shape
    w = inputs.ReduceScatterWorkload(f"rs_r{R}_m{M}_k{K}_n{N}", R, rank, M, K, N, 40 + R)
    x = inputs.make_reduce_scatter_inputs(w)
    _rs_check(w, _rs_dev(x), x)


def test_reduce_scatter_full_size():
    """The benchmark's reduce-scatter workload (rank 1 of 4, 2048 x 4096 x 4096) in full."""
    w = inputs.RS_WORKLOADS[1]
    x = inputs.make_reduce_scatter_inputs(w)
    _rs_check(w, _rs_dev(x), x)


def test_reduce_scatter_new_send_pointers_and_repeat():
    w = inputs.RS_WORKLOADS[0]
    x = inputs.make_reduce_scatter_inputs(w)
    dev = _rs_dev(x)
    with mxa2a.ReduceScatterPlan(w.R, w.rank, w.M, w.K, w.N) as p:
        a = _rs_run(p, dev, w, True)
        b = _rs_run(p, dev, w, True)     # new send buffers: the send maps are re-encoded
    for j in a[0]:
        assert np.array_equal(a[0][j], b[0][j])
    assert np.array_equal(a[1], b[1])


def test_reduce_scatter_argument_errors():
    w = inputs.RS_WORKLOADS[0]
    x = inputs.make_reduce_scatter_inputs(w)
    A, S, B, Bs, recv = _rs_dev(x)
    send = [None if j == w.rank else torch.empty((w.rows, w.N), dtype=torch.int16, device="cuda")
            for j in range(w.R)]
    out = torch.empty((w.rows, w.N), dtype=torch.int16, device="cuda")
    with mxa2a.ReduceScatterPlan(w.R, w.rank, w.M, w.K, w.N) as p:
        C = torch.empty((w.M, w.N), dtype=torch.int16, device="cuda")
        with pytest.raises(mxa2a.Mxa2aError) as e:      # the all-to-all call on this kind
            mxa2a.mxa2a_run(p.handle, [A], [S], B, Bs, C)
        assert e.value.code == mxa2a.MXA2A_ERR_INVALID_OPTION
        bad_recv = list(recv)
        bad_recv[(w.rank + 1) % w.R] = None
        with pytest.raises(mxa2a.Mxa2aError) as e:
            p.run(A, S, B, Bs, bad_recv, send, out)
        assert e.value.code == mxa2a.MXA2A_ERR_NULL_PTR
        flat = torch.empty(w.rows * w.N + 8, dtype=torch.int16, device="cuda")
        bad_send = list(send)
        bad_send[(w.rank + 1) % w.R] = flat.data_ptr() + 2          # 2-byte aligned
        with pytest.raises(mxa2a.Mxa2aError) as e:
            p.run(A, S, B, Bs, recv, bad_send, out)
        assert e.value.code == mxa2a.MXA2A_ERR_MISALIGNED
        torch.cuda.synchronize()
        _status_ok(p)
    with pytest.raises(mxa2a.Mxa2aError):
        mxa2a.ReduceScatterPlan(3, 3, 384, 384, 272)            # rank out of range


# --- GEMM + AllReduce (one-shot) -----------------------------------------------------

def _ar_run(p, dev, w, fused):
    A, S, B, Bs, recv = dev
    pub = torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda")
    out = torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda")
    (p.run if fused else p.run_unfused)(A, S, B, Bs, recv, pub, out)
    torch.cuda.synchronize()
    _status_ok(p)
    return gu.host_bits(pub), gu.host_bits(out)


def _ar_check(w):
    x = inputs.make_allreduce_inputs(w)
    dev = _rs_dev(x)
    with mxa2a.AllReducePlan(w.R, w.rank, w.M, w.K, w.N) as p:
        p.set_option(mxa2a.MXA2A_OPT_TIMEOUT_NS, 500_000_000)
        assert p.get_option(mxa2a.MXA2A_INFO_KIND) == mxa2a.MXA2A_KIND_ALLREDUCE
        pub_f, out_f = _ar_run(p, dev, w, True)
        pub_u, out_u = _ar_run(p, dev, w, False)
    pub_r, out_r = oracle.gemm_allreduce(x["A"], x["A_scale"], x["B"], x["B_scale"],
                                         [None if r is None else r.numpy() for r in x["recv"]], w.R, w.rank)
    gu.assert_parity(pub_f, pub_r, f"{w.name} pub")
    _assert_out_parity(out_f, out_r, pub_r, f"{w.name} out")
    assert np.array_equal(pub_f, pub_u), "pub fused != unfused"
    assert np.array_equal(out_f, out_u), "out fused != unfused"


@pytest.mark.parametrize("w", [inputs.AR_WORKLOADS[0],
                               inputs.AllReduceWorkload("ar_r2_m320_k256_n528", 2, 0, 320, 256, 528, 52),
                               inputs.AllReduceWorkload("ar_r5_m128_k128_n64", 5, 4, 128, 128, 64, 53),
                               inputs.AllReduceWorkload("ar_r1_m64_k256_n256", 1, 0, 64, 256, 256, 54)],
                         ids=lambda w: w.name)
def test_allreduce_small_against_oracle(w):
    _ar_check(w)


def test_allreduce_full_size():
    """The benchmark's all-reduce workload (rank 1 of 4, 2048 x 4096 x 4096) in full."""
    _ar_check(inputs.AR_WORKLOADS[1])


def test_allreduce_argument_errors():
    w = inputs.AR_WORKLOADS[0]
    x = inputs.make_allreduce_inputs(w)
    A, S, B, Bs, recv = _rs_dev(x)
    pub = torch.empty((w.M, w.N), dtype=torch.int16, device="cuda")
    out = torch.empty((w.M, w.N), dtype=torch.int16, device="cuda")
    with mxa2a.AllReducePlan(w.R, w.rank, w.M, w.K, w.N) as p:
        bad = list(recv)
        bad[(w.rank + 1) % w.R] = None
        with pytest.raises(mxa2a.Mxa2aError) as e:
            p.run(A, S, B, Bs, bad, pub, out)
        assert e.value.code == mxa2a.MXA2A_ERR_NULL_PTR
        with pytest.raises(mxa2a.Mxa2aError) as e:      # the reduce-scatter call on this kind
            mxa2a.mxa2a_run_reduce_scatter(p.handle, A, S, B, Bs, recv, [None] * w.R, out)
        assert e.value.code in (mxa2a.MXA2A_ERR_INVALID_OPTION, mxa2a.MXA2A_ERR_NULL_PTR)
        torch.cuda.synchronize()
        _status_ok(p)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_sibling_shapes(seed):
    """Seeded shapes for the three sibling operators against their oracles."""
    rng = np.random.default_rng(700 + seed)
    R = int(rng.integers(1, 6))
    rows = 64 * int(rng.integers(1, 5))
    K = 128 * int(rng.integers(1, 5))
    N = 16 * int(rng.integers(1, 40))
    cm = 64 * int(rng.integers(1, 3))
    if rows % cm:
        cm = 64
    bn = 2
    ag = inputs.AllGatherWorkload("ag_sweep", R, rows, K, N, cm, bn, 710 + seed)
    x = inputs.make_allgather_inputs(ag)
    with _ag_plan(ag) as p:
        got_f = _ag_run(p, _ag_dev(x), ag.M, ag.N, "fused")
        got_u = _ag_run(p, _ag_dev(x), ag.M, ag.N, "unfused")
    gu.assert_parity(got_f, oracle.gemm_allgather(x["A_blk"], x["A_scale_blk"], x["B"], x["B_scale"]), "ag sweep")
    assert np.array_equal(got_f, got_u)
    rank = int(rng.integers(0, R))
    rs = inputs.ReduceScatterWorkload("rs_sweep", R, rank, R * rows, K, N, 720 + seed)
    xr = inputs.make_reduce_scatter_inputs(rs)
    _rs_check(rs, _rs_dev(xr), xr)
    _ar_check(inputs.AllReduceWorkload("ar_sweep", R, rank, rows, K, N, 730 + seed))
