"""Failure detection without a GPU fault: a staging step that is never
published makes the bounded device waits run out; the kernel reports
MXA2A_ERR_TIMEOUT through the status block, leaves the context usable, and
the next run is correct.  (The pages' playbook for lost signals, performance
guide 2.1: a slot whose producer never notifies leaves its consumers waiting.)"""
import numpy as np
import pytest
import torch

from all_mxfp8_block_gb300 import inputs, mxa2a
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from all_mxfp8_block_gb300 import build
    build.build()
    mxa2a.load()
    torch.cuda.init()


@pytest.mark.parametrize("split,skip", [(1, 3), (2, 3), (1, 0)])
def test_lost_staging_signal_times_out_then_recovers(split, skip):
    """skip 3: a step in the middle never comes; skip 0: the first one, so
    every producer gives up before its first load."""
    w = inputs.Workload("fault", 2, 512, 256, 512, 64, 2, 53)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num) as p:
        p.set_option(mxa2a.MXA2A_OPT_TIMEOUT_NS, 100_000_000)      # 0.1 s per wait
        p.set_option(mxa2a.MXA2A_OPT_SPLIT_K, split)
        p.set_option(mxa2a.MXA2A_OPT_FAULT_SKIP_STEP, skip)
        gu.run_gpu(p, d, w.M, w.N)
        torch.cuda.synchronize()                                      # returns: every wait is bounded
        st = p.status()
        assert st["code"] == mxa2a.MXA2A_ERR_TIMEOUT, st
        assert st["launch"] >= 1
        # the context is intact and the credits were reset by the last CTA
        assert np.all(p.read_workspace(mxa2a.MXA2A_WS_FLAGS).view(np.uint64) == 0)
        p.set_option(mxa2a.MXA2A_OPT_FAULT_SKIP_STEP, -1)
        C = gu.run_gpu(p, d, w.M, w.N)
        torch.cuda.synchronize()
        assert p.status()["code"] == 0
        got = gu.host_bits(C)
    gu.assert_parity(got, gu.oracle_full(x), f"after recovery split={split} skip={skip}")


def test_lost_staging_signal_cta_pair():
    """The same on the fused CTA-pair kernel: both CTAs of every pair give up
    through their bounded waits, the even CTA completes the stages only one of
    them armed or loaded, both meet at the cluster barriers, and the next run
    on the plan is correct."""
    w = inputs.Workload("faultpair", 2, 512, 256, 512, 128, 2, 57)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num) as p:
        p.set_option(mxa2a.MXA2A_OPT_TIMEOUT_NS, 100_000_000)
        p.set_option(mxa2a.MXA2A_OPT_CTA_PAIR, 1)
        p.set_option(mxa2a.MXA2A_OPT_SPLIT_K, 1)
        assert p.get_option(mxa2a.MXA2A_INFO_CTA_PAIR) == 1
        p.set_option(mxa2a.MXA2A_OPT_FAULT_SKIP_STEP, 3)
        gu.run_gpu(p, d, w.M, w.N)
        torch.cuda.synchronize()
        st = p.status()
        assert st["code"] == mxa2a.MXA2A_ERR_TIMEOUT, st
        assert np.all(p.read_workspace(mxa2a.MXA2A_WS_FLAGS).view(np.uint64) == 0)
        p.set_option(mxa2a.MXA2A_OPT_FAULT_SKIP_STEP, -1)
        C = gu.run_gpu(p, d, w.M, w.N)
        torch.cuda.synchronize()
        assert p.status()["code"] == 0
        got = gu.host_bits(C)
    gu.assert_parity(got, gu.oracle_full(x), "after recovery, CTA pairs")


def test_status_is_clean_after_normal_runs():
    w = inputs.workload(0)
    x = inputs.make_inputs(w)
    d = gu.to_device(x)
    with mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num) as p:
        for _ in range(3):
            gu.run_gpu(p, d, w.M, w.N)
        torch.cuda.synchronize()
        st = p.status()
    assert st["code"] == 0 and st["step"] == -1
