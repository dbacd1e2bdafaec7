"""The allocation-free entry point, mxa2a_run_noalloc.

It serves callers that cannot allocate device memory (a runtime whose device
memory is all owned by its own pool allocator, or a latency-critical loop in
which cudaMalloc / cudaFree would synchronise the device): its scratch is a
static 16 MiB device array inside the library instead of a plan's workspace.
The GPU test calls it twice in a row through the C ABI, on two different
problems, and checks each result against mxa2a_run's within the parity
tolerance the other GPU tests use.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from all_mxfp8_block_gb300 import inputs, mxa2a


def test_noalloc_rejects_problems_larger_than_its_scratch():
    from all_mxfp8_block_gb300 import build
    build.build()
    lib = mxa2a.load()
    # the 8 x 8192 x 8192 x 8192 workload needs a 16 MiB ring plus 4 MiB of scale tiles
    w = inputs.workload(3)
    rc = lib.mxa2a_run_noalloc(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num,
                               None, None, None, None, None, None)
    assert rc == mxa2a.MXA2A_ERR_SCRATCH_TOO_SMALL
    assert "scratch" in mxa2a.strerror(rc)
    # shape rules come first
    assert lib.mxa2a_run_noalloc(2, 100, 128, 256, 64, 2, None, None, None, None, None, None) == \
        mxa2a.MXA2A_ERR_INVALID_SHAPE


def _device_inputs(w):
    x = inputs.make_inputs(w)
    return {"A_seg": [a.cuda() for a in x["A_seg"]], "A_scale_seg": [s.cuda() for s in x["A_scale_seg"]],
            "B": x["B"].cuda(), "B_scale": x["B_scale"].cuda()}


def _reference_with_plan(w, d):
    C = torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda")
    with mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num) as p:
        p.run(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C)
        torch.cuda.synchronize()
        assert p.status()["code"] == 0
    return C


def _within_tolerance(got, ref):
    g = (got.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (ref.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert not np.isnan(g).any()
    bad = np.abs(g - r) > 1e-2 + 1e-2 * np.abs(r)
    return int(bad.sum())


@pytest.mark.gpu
def test_noalloc_matches_plan_entry_on_two_calls_in_a_row():
    from all_mxfp8_block_gb300 import build
    build.build()
    mxa2a.load()
    torch.cuda.init()
    problems = [inputs.workload(1), inputs.workload(0)]      # 4 x 2048 x 4096 x 4096, then the tiny one
    data = [_device_inputs(w) for w in problems]
    refs = [_reference_with_plan(w, d) for w, d in zip(problems, data)]
    outs = []
    for w, d in zip(problems, data):                         # two calls back to back, one stream
        C = torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda")
        mxa2a.mxa2a_run_noalloc(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num,
                                d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C)
        outs.append(C)
    torch.cuda.synchronize()
    for w, got, ref in zip(problems, outs, refs):
        assert _within_tolerance(got, ref) == 0, w.name
