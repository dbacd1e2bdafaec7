"""Seeded synthetic MXFP8 inputs for the fused AllToAll + block-scaled GEMM.

This module only draws random numbers and quantises them into the byte
format the operation consumes; it holds none of the operation's arithmetic
(no decoding, no products, no accumulation).  Both the CUDA path's tests and
the CPU oracle's tests take their inputs from here.

Operand format (the MX "FP8" format named by the all_to_all_matmul kernel
entry, ``AllToAllQuantMatmulKernelE4M3E4M3``, with ``fp8_e4m3fn_t`` data and
``fp8_e8m0_t`` scales, all_to_all_matmul_impl.h):

* ``A_seg[r]``      uint8 ``[M][kPerRank]``   E4M3 codes of segment ``r``
* ``A_scale_seg[r]``uint8 ``[M][kPerRank/32]`` E8M0 scale bytes, one per 32 along K
* ``B``             uint8 ``[N][K]``          E4M3 codes, stored transposed
  (the kernel is instantiated with ``TransB=true``), ``K = R * kPerRank``
* ``B_scale``       uint8 ``[N][K/32]``       E8M0 scale bytes

The quantiser follows the OCP MX recipe: per 32-element block the shared
exponent is ``floor(log2(amax)) - 8`` (8 = largest E4M3 exponent), clamped to
the E8M0 range; elements are divided by it, saturated to +-448 and rounded to
nearest-even by ``torch``'s own float8 conversion.  An all-zero block gets
scale byte 0 and zero codes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

MX_BLOCK = 32          # elements per E8M0 scale along K
E4M3_EMAX = 8          # exponent of the largest E4M3 binade (448 = 1.75 * 2^8)
E4M3_MAX = 448.0
E5M2_EMAX = 15         # exponent of the largest E5M2 binade (57344 = 1.75 * 2^15)
E5M2_MAX = 57344.0
# element formats: (largest binade exponent, largest value, torch dtype)
FORMATS = {"e4m3": (E4M3_EMAX, E4M3_MAX, torch.float8_e4m3fn),
           "e5m2": (E5M2_EMAX, E5M2_MAX, torch.float8_e5m2)}


@dataclass(frozen=True)
class Workload:
    """One problem size of the fused AllToAll + MXFP8 GEMM."""
    name: str
    R: int            # number of K segments ("ranks")
    M: int            # rows of A and C
    kPerRank: int     # K extent of one segment
    N: int            # columns of C
    commMSize: int    # rows per staging step
    buffer_num: int   # staging ring depth
    seed: int
    outliers: bool = False   # 1% x100 rows and 2^-6..2^6 per-block spread on A
    note: str = field(default="", compare=False)
    a_fmt: str = "e4m3"      # element format of A ("e4m3" or "e5m2")
    b_fmt: str = "e4m3"      # element format of B

    @property
    def K(self) -> int:
        return self.R * self.kPerRank

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_alg(self) -> int:
        """Bytes the operation must move once: A, its scales, B, its scales, C."""
        K = self.K
        return (self.M * K + self.M * K // MX_BLOCK + self.N * K
                + self.N * K // MX_BLOCK + 2 * self.M * self.N)


# The five problem sizes the method is exercised on.  The first is the small
# case the CPU oracle finishes in well under a second; the second is the one
# the headline throughput is quoted on.
WORKLOADS = [
    Workload("r2_m128_k256_n256", 2, 128, 128, 256, 64, 2, 0,
             note="tiny: two 64-row staging steps, one output tile"),
    Workload("r4_m2048_k4096_n4096", 4, 2048, 1024, 4096, 256, 2, 1,
             note="square-ish, tensor-core bound"),
    Workload("r8_m4096_k7168_n2048", 8, 4096, 896, 2048, 512, 4, 2,
             note="MoE-projection-like shape"),
    Workload("r8_m8192_k8192_n8192", 8, 8192, 1024, 8192, 512, 4, 3,
             note="compute-bound"),
    Workload("r16_m64_k8192_n7168", 16, 64, 512, 7168, 64, 2, 4, outliers=True,
             note="small M: HBM bound on B, needs split-K to fill the GPU"),
]
WORKLOADS_BY_NAME = {w.name: w for w in WORKLOADS}


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    return WORKLOADS_BY_NAME[name_or_index]


def quantize_mx_rows(x: torch.Tensor, fmt: str = "e4m3") -> tuple[torch.Tensor, torch.Tensor]:
    """Quantise fp32 ``[rows][K]`` (K % 32 == 0) to (element codes, E8M0 bytes),
    OCP MX: per 32-block X = floor(log2 amax) - emax of the element format,
    elements = round-to-nearest-even of clamp(v / 2^X, +-max).

    Returns ``codes`` uint8 ``[rows][K]`` and ``scales`` uint8 ``[rows][K/32]``.
    """
    emax, vmax, dtype = FORMATS[fmt]
    assert x.dtype == torch.float32 and x.dim() == 2 and x.shape[1] % MX_BLOCK == 0
    rows, K = x.shape
    blocks = x.reshape(rows, K // MX_BLOCK, MX_BLOCK)
    amax = blocks.abs().amax(dim=2)
    # frexp: amax = mant * 2^e with mant in [0.5, 1)  =>  floor(log2 amax) = e - 1
    _, e = torch.frexp(amax)
    X = (e.to(torch.int32) - 1) - emax
    X = torch.where(amax > 0, X, torch.full_like(X, -127))
    X = X.clamp(-127, 127)
    scaled = torch.ldexp(blocks, (-X).to(torch.float32).unsqueeze(2))
    scaled = scaled.clamp(-vmax, vmax)
    codes = scaled.to(dtype).view(torch.uint8).reshape(rows, K)
    scales = (X + 127).to(torch.uint8)
    return codes.contiguous(), scales.contiguous()


def make_inputs(w: Workload) -> dict:
    """Draw and quantise the inputs of workload ``w`` (CPU tensors).

    Draw order with ``torch.Generator().manual_seed(seed)``: ``A_r =
    randn(M, kPerRank)`` for r = 0..R-1; for the outlier workload the row
    permutation and the per-block exponent spread; then ``B = randn(K, N) /
    sqrt(K)``.
    """
    g = torch.Generator().manual_seed(w.seed)
    A = [torch.randn(w.M, w.kPerRank, generator=g, dtype=torch.float32)
         for _ in range(w.R)]
    if w.outliers:
        n_out = max(1, int(round(0.01 * w.M)))
        rows = torch.randperm(w.M, generator=g)[:n_out]
        u = torch.randint(-6, 7, (w.M, w.K // MX_BLOCK), generator=g)
        mult = torch.pow(2.0, u.to(torch.float32))
        full = torch.cat(A, dim=1)
        full[rows] *= 100.0
        full = (full.reshape(w.M, w.K // MX_BLOCK, MX_BLOCK)
                * mult.unsqueeze(2)).reshape(w.M, w.K)
        A = list(full.split(w.kPerRank, dim=1))
    B = torch.randn(w.K, w.N, generator=g, dtype=torch.float32) / math.sqrt(w.K)
    A_seg, A_sf = [], []
    for a in A:
        c, s = quantize_mx_rows(a.contiguous(), w.a_fmt)
        A_seg.append(c)
        A_sf.append(s)
    B_codes, B_sf = quantize_mx_rows(B.t().contiguous(), w.b_fmt)
    return {"A_seg": A_seg, "A_scale_seg": A_sf, "B": B_codes, "B_scale": B_sf,
            "workload": w}


def make_custom(R: int, M: int, kPerRank: int, N: int, seed: int,
                commMSize: int = 64, buffer_num: int = 2) -> dict:
    """Inputs for an ad-hoc shape, drawn exactly like :func:`make_inputs`."""
    w = Workload(f"custom_r{R}_m{M}_ka{kPerRank}_n{N}", R, M, kPerRank, N,
                 commMSize, buffer_num, seed)
    return make_inputs(w)


def random_codes(shape, seed: int, allow_nan: bool = False) -> torch.Tensor:
    """Uniformly random E4M3 code bytes (subnormals included); NaN codes
    0x7F/0xFF are replaced by +-448 unless ``allow_nan``."""
    g = torch.Generator().manual_seed(seed)
    c = torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(torch.uint8)
    if not allow_nan:
        c = torch.where(c == 0x7F, torch.tensor(0x7E, dtype=torch.uint8), c)
        c = torch.where(c == 0xFF, torch.tensor(0xFE, dtype=torch.uint8), c)
    return c


def random_scales(shape, seed: int, lo: int = 0, hi: int = 254) -> torch.Tensor:
    """Uniformly random E8M0 scale bytes in ``[lo, hi]`` (255 = NaN excluded)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int32).to(torch.uint8)


# --- the sibling fused operators ------------------------------------------------------

@dataclass(frozen=True)
class AllGatherWorkload:
    """One problem size of AllGather + GEMM: R row blocks of rowsPerRank rows
    (all K columns) stacked along M, times B [N][K]."""
    name: str
    R: int
    rowsPerRank: int
    K: int
    N: int
    commMSize: int
    buffer_num: int
    seed: int

    @property
    def M(self) -> int:
        return self.R * self.rowsPerRank

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_alg(self) -> int:
        M, K, N = self.M, self.K, self.N
        return M * K + M * K // MX_BLOCK + N * K + N * K // MX_BLOCK + 2 * M * N


@dataclass(frozen=True)
class ReduceScatterWorkload:
    """One problem size of GEMM + ReduceScatter, seen from rank ``rank`` of
    ``R``: A [M][K], B [N][K], blocks of M / R rows."""
    name: str
    R: int
    rank: int
    M: int
    K: int
    N: int
    seed: int

    @property
    def rows(self) -> int:
        return self.M // self.R

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_alg(self) -> int:
        """A, B and their scales once; R-1 received blocks, R-1 sent blocks and the output block (BF16)."""
        M, K, N = self.M, self.K, self.N
        return (M * K + M * K // MX_BLOCK + N * K + N * K // MX_BLOCK
                + 2 * (2 * (self.R - 1) + 1) * self.rows * N)


# The sibling workloads: a small one the oracle finishes at once, and one of
# the headline's size (2048 x 4096 x 4096 flops, 4 ranks; the all-gather's
# ring holds two 256-row steps, as the headline all-to-all's does).
AG_WORKLOADS = [
    AllGatherWorkload("ag_r3_m384_k384_n272", 3, 128, 384, 272, 64, 2, 20),
    AllGatherWorkload("ag_r4_m2048_k4096_n4096", 4, 512, 4096, 4096, 256, 2, 21),
]
RS_WORKLOADS = [
    ReduceScatterWorkload("rs_r3_m384_k384_n272", 3, 1, 384, 384, 272, 30),
    ReduceScatterWorkload("rs_r4_m2048_k4096_n4096", 4, 1, 2048, 4096, 4096, 31),
]


@dataclass(frozen=True)
class AllReduceWorkload:
    """One problem size of GEMM + AllReduce (one-shot), seen from rank
    ``rank`` of ``R``: A [M][K], B [N][K]; every rank ends with the sum of
    all ranks' [M][N] partials."""
    name: str
    R: int
    rank: int
    M: int
    K: int
    N: int
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_alg(self) -> int:
        """A, B and their scales once; R-1 peers' partials read; the published partial and out written (BF16)."""
        M, K, N = self.M, self.K, self.N
        return M * K + M * K // MX_BLOCK + N * K + N * K // MX_BLOCK + 2 * (self.R + 1) * M * N


AR_WORKLOADS = [
    AllReduceWorkload("ar_r3_m192_k384_n272", 3, 1, 192, 384, 272, 50),
    AllReduceWorkload("ar_r4_m2048_k4096_n4096", 4, 1, 2048, 4096, 4096, 51),
]


def make_allgather_inputs(w: AllGatherWorkload) -> dict:
    """Draw and quantise AllGather + GEMM inputs (CPU tensors).  Draw order:
    ``A_j = randn(rowsPerRank, K)`` for j = 0..R-1, then ``B = randn(K, N) /
    sqrt(K)``."""
    g = torch.Generator().manual_seed(w.seed)
    A = [torch.randn(w.rowsPerRank, w.K, generator=g, dtype=torch.float32) for _ in range(w.R)]
    B = torch.randn(w.K, w.N, generator=g, dtype=torch.float32) / math.sqrt(w.K)
    A_blk, A_sf = [], []
    for a in A:
        c, s = quantize_mx_rows(a.contiguous())
        A_blk.append(c)
        A_sf.append(s)
    B_codes, B_sf = quantize_mx_rows(B.t().contiguous())
    return {"A_blk": A_blk, "A_scale_blk": A_sf, "B": B_codes, "B_scale": B_sf, "workload": w}


def make_reduce_scatter_inputs(w: ReduceScatterWorkload) -> dict:
    """Draw GEMM + ReduceScatter inputs (CPU tensors).  Draw order: ``A =
    randn(M, K)``, ``B = randn(K, N) / sqrt(K)`` (quantised to MXFP8 as for
    the all-to-all), then for every peer j != rank in order the partial it
    sent, ``randn(M/R, N)`` rounded to BF16 (the magnitude of a partial of
    this shape), as int16 bit patterns; ``recv[rank]`` is None."""
    g = torch.Generator().manual_seed(w.seed)
    A = torch.randn(w.M, w.K, generator=g, dtype=torch.float32)
    B = torch.randn(w.K, w.N, generator=g, dtype=torch.float32) / math.sqrt(w.K)
    recv = []
    for j in range(w.R):
        if j == w.rank:
            recv.append(None)
        else:
            r = torch.randn(w.rows, w.N, generator=g, dtype=torch.float32)
            recv.append(r.to(torch.bfloat16).view(torch.int16).contiguous())
    A_codes, A_sf = quantize_mx_rows(A)
    B_codes, B_sf = quantize_mx_rows(B.t().contiguous())
    return {"A": A_codes, "A_scale": A_sf, "B": B_codes, "B_scale": B_sf, "recv": recv, "workload": w}


def make_allreduce_inputs(w: AllReduceWorkload) -> dict:
    """Draw GEMM + AllReduce inputs (CPU tensors).  Draw order: ``A =
    randn(M, K)``, ``B = randn(K, N) / sqrt(K)`` (quantised to MXFP8), then
    for every peer j != rank in order its published partial ``randn(M, N)``
    rounded to BF16, as int16 bit patterns; ``recv[rank]`` is None."""
    g = torch.Generator().manual_seed(w.seed)
    A = torch.randn(w.M, w.K, generator=g, dtype=torch.float32)
    B = torch.randn(w.K, w.N, generator=g, dtype=torch.float32) / math.sqrt(w.K)
    recv = []
    for j in range(w.R):
        if j == w.rank:
            recv.append(None)
        else:
            r = torch.randn(w.M, w.N, generator=g, dtype=torch.float32)
            recv.append(r.to(torch.bfloat16).view(torch.int16).contiguous())
    A_codes, A_sf = quantize_mx_rows(A)
    B_codes, B_sf = quantize_mx_rows(B.t().contiguous())
    return {"A": A_codes, "A_scale": A_sf, "B": B_codes, "B_scale": B_sf, "recv": recv, "workload": w}
