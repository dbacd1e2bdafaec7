"""Helpers shared by the GPU tests: device copies of the seeded inputs, runs
through the C ABI, and the parity report against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from all_mxfp8_block_gb300 import inputs, mxa2a

ATOL = 1e-2
RTOL = 1e-2


def to_device(x: dict, device="cuda") -> dict:
    return {
        "A_seg": [a.to(device) for a in x["A_seg"]],
        "A_scale_seg": [s.to(device) for s in x["A_scale_seg"]],
        "B": x["B"].to(device),
        "B_scale": x["B_scale"].to(device),
    }


def run_gpu(plan: mxa2a.Plan, d: dict, M: int, N: int, fused=True, stream=None) -> torch.Tensor:
    """One run; fused True = mxa2a_run, False = mxa2a_run_unfused, "direct" = mxa2a_run_direct."""
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")   # 0xFFFF: a BF16 NaN until written
    fn = plan.run_direct if fused == "direct" else (plan.run if fused else plan.run_unfused)
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())   # inputs and C were written on it
    fn(d["A_seg"], d["A_scale_seg"], d["B"], d["B_scale"], C, stream)
    return C


def host_bits(C) -> np.ndarray:
    """BF16 bit patterns of a device int16 [M][N] tensor as a uint16 numpy array."""
    return C.cpu().numpy().view(np.uint16)


def bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits).view(np.uint16) if np.asarray(bits).dtype == np.int16 else np.asarray(bits, dtype=np.uint16)
    return oracle.bf16_bits_to_f32(b).astype(np.float64)


def parity_stats(gpu_bits, ref_bits) -> dict:
    """The pages' verify report (max/mean abs error, RMSE, max rel error with the
    denominator clamped at 1e-8, count above 1e-2) plus the per-element gate
    |gpu - ref| <= ATOL + RTOL*|ref| (and the pages' allclose form |..| <= ATOL + RTOL*|gpu|)."""
    g = bits_to_f64(gpu_bits)
    r = bits_to_f64(ref_bits)
    nan_g, nan_r = np.isnan(g), np.isnan(r)
    # an infinity matches the same infinity exactly (inf - inf would be NaN);
    # an infinity against anything else fails the gate below
    same_inf = np.isinf(g) & np.isinf(r) & (g == r)
    inf_mismatch = (np.isinf(g) | np.isinf(r)) & ~same_inf & ~(nan_g | nan_r)
    both = ~(nan_g | nan_r | same_inf | inf_mismatch)
    diff = g[both] - r[both]
    ad = np.abs(diff)
    rel = ad / np.maximum(np.abs(r[both]), 1e-8)
    gate = ad <= ATOL + RTOL * np.abs(r[both])
    gate_pages = ad <= ATOL + RTOL * np.abs(g[both])
    return {
        "n": int(g.size),
        "max_abs": float(ad.max()) if ad.size else 0.0,
        "mean_abs": float(ad.mean()) if ad.size else 0.0,
        "rmse": float(np.sqrt((diff ** 2).mean())) if ad.size else 0.0,
        "max_rel": float(rel.max()) if rel.size else 0.0,
        "over_1e-2": int((ad > 1e-2).sum()),
        "fail": int((~gate).sum()) + int((nan_g != nan_r).sum()) + int(inf_mismatch.sum()),
        "inf_matched": int(same_inf.sum()),
        "inf_mismatch": int(inf_mismatch.sum()),
        "fail_pages_form": int((~gate_pages).sum()),
        "nan_mismatch": int((nan_g != nan_r).sum()),
    }


def assert_parity(gpu_bits, ref_bits, label=""):
    st = parity_stats(gpu_bits, ref_bits)
    print(f"[parity] {label} {st}")
    assert st["fail"] == 0, (label, st)
    return st


def oracle_full(x: dict) -> np.ndarray:
    w = x.get("workload")
    fmts = {"a_fmt": w.a_fmt, "b_fmt": w.b_fmt} if w is not None else {}
    return oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"], **fmts)


def sample_rows(M: int, n: int, seed: int) -> np.ndarray:
    """n rows spread over M: the first and last row of every 128-row tile hit, plus random ones."""
    rng = np.random.default_rng(seed)
    fixed = {0, M - 1, min(M - 1, 127), min(M - 1, 128), M // 2}
    rest = rng.choice(M, size=max(0, n - len(fixed)), replace=False)
    return np.array(sorted(fixed | set(int(v) for v in rest)), dtype=np.int64)
