"""The seeded input generator: deterministic, and a faithful MX quantiser."""
import numpy as np
import torch

from all_mxfp8_block_gb300 import inputs
from tests import _exact


def test_generator_is_deterministic():
    w = inputs.workload(0)
    a, b = inputs.make_inputs(w), inputs.make_inputs(w)
    for k in ("A_seg", "A_scale_seg"):
        for x, y in zip(a[k], b[k]):
            assert torch.equal(x, y)
    assert torch.equal(a["B"], b["B"]) and torch.equal(a["B_scale"], b["B_scale"])


def test_shapes_and_dtypes():
    w = inputs.workload(0)
    x = inputs.make_inputs(w)
    assert len(x["A_seg"]) == w.R
    for a, s in zip(x["A_seg"], x["A_scale_seg"]):
        assert a.shape == (w.M, w.kPerRank) and a.dtype == torch.uint8
        assert s.shape == (w.M, w.kPerRank // 32) and s.dtype == torch.uint8
    assert x["B"].shape == (w.N, w.K) and x["B_scale"].shape == (w.N, w.K // 32)


def test_quantiser_reconstructs_within_e4m3_precision():
    g = torch.Generator().manual_seed(3)
    v = torch.randn(64, 256, generator=g) * torch.pow(2.0, torch.randint(-20, 20, (64, 1), generator=g).float())
    codes, sc = inputs.quantize_mx_rows(v)
    q = _exact.e4m3_values(codes.numpy()) * np.repeat(_exact.e8m0_values(sc.numpy()), 32, axis=1)
    vv = v.double().numpy()
    blocks = np.abs(vv).reshape(64, 8, 32).max(axis=2)
    # block maximum lands in [256, 448] after scaling (448 is the saturation point)
    scaled_max = blocks / _exact.e8m0_values(sc.numpy())
    assert np.all((scaled_max >= 256) & (scaled_max < 512))
    # elements: half-ulp of E4M3 (2^-4 relative) or half the subnormal step
    step = np.repeat(_exact.e8m0_values(sc.numpy()), 32, axis=1) * 2.0 ** -10
    err = np.abs(q - vv)
    tol = np.maximum(np.abs(vv) * 2.0 ** -4, step) + np.maximum(np.abs(vv) - 448 * np.repeat(_exact.e8m0_values(sc.numpy()), 32, axis=1), 0)
    assert np.all(err <= tol * (1 + 1e-12))


def test_outlier_workload_spreads_block_exponents():
    w = inputs.workload(4)
    x = inputs.make_inputs(w)
    s = torch.cat(x["A_scale_seg"], dim=1).int()
    assert int(s.max() - s.min()) >= 12          # 2^-6..2^6 spread plus the x100 rows
    assert x["A_seg"][0].shape == (64, 512)
