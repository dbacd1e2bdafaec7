"""The allocation-free entry point, mxa2a_run_noalloc.

It serves callers that cannot allocate device memory (a runtime whose device
memory is all owned by its own pool allocator, or a latency-critical loop in
which cudaMalloc / cudaFree would synchronise the device): its scratch is a
static 16 MiB device array inside the library instead of a plan's workspace.

The GPU test calls it three times in a row through the C ABI, on three
problems, and checks each result bit for bit against mxa2a_run of a plan
forced to the same (unsplit) K loop, and against the oracle on sampled rows
within the parity tolerance of the other GPU tests.  The 64-row problem
follows a 2048-row one, so the scale tiles of its rows past M are stale in the
shared array unless the entry point clears them.  It also checks that the
calls allocate nothing on the device.  This file is collected last on purpose.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
from all_mxfp8_block_gb300 import inputs, mxa2a
from tests import gpu_util as gu


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


def _reference_with_plan(w, d):
    """mxa2a_run of a plan on the entry point's kernel: the single-CTA kernel,
    K loop not split (the last round's tiles neither)."""
    C = torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda")
    with mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num) as p:
        p.set_option(mxa2a.MXA2A_OPT_SPLIT_K, 1)
        p.set_option(mxa2a.MXA2A_OPT_CTA_PAIR, 0)
        p.set_option(mxa2a.MXA2A_OPT_TAIL_SPLIT, 0)
        p.run(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C)
        torch.cuda.synchronize()
        assert p.status()["code"] == 0
    return C


@pytest.mark.gpu
def test_noalloc_matches_plan_entry_on_calls_in_a_row():
    from all_mxfp8_block_gb300 import build
    build.build()
    mxa2a.load()
    torch.cuda.init()
    # 4 x 2048 x 4096 x 4096, then 16 x 64 x 8192 x 7168 (rows past M in its only
    # m-tile), then the tiny one
    problems = [inputs.workload(1), inputs.workload(4), inputs.workload(0)]
    host = [inputs.make_inputs(w) for w in problems]
    data = [gu.to_device(x) for x in host]
    refs = [_reference_with_plan(w, d) for w, d in zip(problems, data)]
    outs = [torch.full((w.M, w.N), -1, dtype=torch.int16, device="cuda") for w in problems]

    def call(i):
        w, d = problems[i], data[i]
        mxa2a.mxa2a_run_noalloc(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num,
                                d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], outs[i])

    # the first call on the device looks up the scratch array's address (once)
    call(2)
    torch.cuda.synchronize()
    gc.collect()   # (earlier tests' tensors are freed now, not during the calls)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    torch_before = torch.cuda.memory_allocated()
    for i in range(len(problems)):                           # back to back, one stream
        call(i)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before, (free_before, free_after)

    for i, (w, x) in enumerate(zip(problems, host)):
        got, ref = gu.host_bits(outs[i]), gu.host_bits(refs[i])
        assert np.array_equal(got, ref), w.name
        rows = gu.sample_rows(w.M, 24 if w.M > 64 else w.M, seed=100 + i)
        exact = oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"], rows=rows)
        gu.assert_parity(got[rows], exact, f"noalloc {w.name} sampled {len(rows)} rows")
