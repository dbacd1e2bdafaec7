"""Thin ctypes binding of libmxa2a (``include/mxa2a.h``): argument marshalling only.

Every function keeps the C name and argument order; tensors are passed as raw
device (or, for ``mxa2a_run_host``, host) pointers taken from ``torch``
tensors or numpy arrays.  Every computation runs inside the library's CUDA
kernels: there is no fallback, and a missing or unloadable ``libmxa2a.so``
raises :class:`Mxa2aError` immediately.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmxa2a.so")

# --- constants mirrored from include/mxa2a.h (a CPU test checks they match) ---
MXA2A_OK = 0
MXA2A_ERR_INVALID_SHAPE = 1
MXA2A_ERR_NULL_PTR = 2
MXA2A_ERR_MISALIGNED = 3
MXA2A_ERR_UNSUPPORTED_DEVICE = 4
MXA2A_ERR_CUDA = 5
MXA2A_ERR_TIMEOUT = 6
MXA2A_ERR_INVALID_OPTION = 7
MXA2A_ERR_DEVICE_CHECK = 8
MXA2A_ERR_WRONG_DEVICE = 9
MXA2A_ERR_SCRATCH_TOO_SMALL = 10
MXA2A_ERR_CAPTURE_SPLIT = 11

MXA2A_OPT_TIMEOUT_NS = 1
MXA2A_OPT_SPLIT_K = 2
MXA2A_OPT_ZIGZAG = 3
MXA2A_OPT_ROTATE = 4
MXA2A_OPT_RECORD_EVENTS = 5
MXA2A_OPT_EXCHANGE_ONLY = 6
MXA2A_OPT_FAULT_SKIP_STEP = 7
MXA2A_OPT_GRID = 8
MXA2A_OPT_CHUNK_BYTES = 9
MXA2A_OPT_CTA_PAIR = 10
MXA2A_OPT_GROUP_M = 11
MXA2A_OPT_TILE_N = 13
MXA2A_OPT_ELEM_TYPES = 14
MXA2A_OPT_STEP_CREDITS = 15
MXA2A_OPT_COPY_SKEW_NS = 16
MXA2A_OPT_GROUP_FUSED = 17
MXA2A_OPT_TAIL_SPLIT = 18
ELEM_TYPES = {("e4m3", "e4m3"): 0, ("e5m2", "e5m2"): 1, ("e4m3", "e5m2"): 2, ("e5m2", "e4m3"): 3}
MXA2A_INFO_STEPS = 100
MXA2A_INFO_MTILES = 101
MXA2A_INFO_NTILES = 102
MXA2A_INFO_SPLITS = 103
MXA2A_INFO_ITEMS = 104
MXA2A_INFO_GRID_FUSED = 105
MXA2A_INFO_GRID_UNFUSED = 106
MXA2A_INFO_COPY_TASKS = 107
MXA2A_INFO_ROWS_PER_CHUNK = 108
MXA2A_INFO_WORKSPACE_BYTES = 109
MXA2A_INFO_SM_COUNT = 110
MXA2A_INFO_LAUNCHES = 111
MXA2A_INFO_SPLITS_UNFUSED = 112
MXA2A_INFO_CTA_PAIR = 113
MXA2A_INFO_CTA_PAIR_UNFUSED = 114
MXA2A_INFO_GROUP_FUSED = 115
MXA2A_INFO_GROUP_UNFUSED = 116
MXA2A_INFO_TILE_N_FUSED = 117
MXA2A_INFO_TILE_N_UNFUSED = 118
MXA2A_INFO_KIND = 119
MXA2A_INFO_TAIL_SPLIT = 120
MXA2A_INFO_TAIL_SPLIT_UNFUSED = 121

MXA2A_KIND_ALLTOALL = 0
MXA2A_KIND_ALLGATHER = 1
MXA2A_KIND_REDUCE_SCATTER = 2
MXA2A_KIND_ALLREDUCE = 3

MXA2A_WS_RING = 1
MXA2A_WS_SFA = 2
MXA2A_WS_SFB = 3
MXA2A_WS_FLAGS = 4
MXA2A_WS_APACKED = 5


class Mxa2aError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})")


class mxa2a_status(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int32), ("role", ctypes.c_int32), ("block", ctypes.c_int32),
                ("step", ctypes.c_int32), ("segment", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("observed", ctypes.c_int64), ("expected", ctypes.c_int64), ("launch", ctypes.c_int64)]


_lib = None

# (name, restype, argtypes) of every exported function
_VP = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)
_I64 = ctypes.c_int64
_SIGS = [
    ("mxa2a_validate", ctypes.c_int, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int]),
    ("mxa2a_create", _VP, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int]),
    ("mxa2a_last_error", ctypes.c_int, []),
    ("mxa2a_validate_allgather", ctypes.c_int, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int]),
    ("mxa2a_create_allgather", _VP, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int]),
    ("mxa2a_validate_reduce_scatter", ctypes.c_int, [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64]),
    ("mxa2a_create_reduce_scatter", _VP, [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64]),
    ("mxa2a_run_reduce_scatter", ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _PP, _PP, _VP, _VP]),
    ("mxa2a_run_reduce_scatter_unfused", ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _PP, _PP, _VP, _VP]),
    ("mxa2a_validate_allreduce", ctypes.c_int, [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64]),
    ("mxa2a_create_allreduce", _VP, [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64]),
    ("mxa2a_run_allreduce", ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _PP, _VP, _VP, _VP]),
    ("mxa2a_run_allreduce_unfused", ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _PP, _VP, _VP, _VP]),
    ("mxa2a_run", ctypes.c_int, [_VP, _PP, _PP, _VP, _VP, _VP, _VP]),
    ("mxa2a_run_unfused", ctypes.c_int, [_VP, _PP, _PP, _VP, _VP, _VP, _VP]),
    ("mxa2a_run_direct", ctypes.c_int, [_VP, _PP, _PP, _VP, _VP, _VP, _VP]),
    ("mxa2a_run_host", ctypes.c_int, [_VP, _PP, _PP, _VP, _VP, _VP, _VP]),
    ("mxa2a_get_status", ctypes.c_int, [_VP, ctypes.POINTER(mxa2a_status)]),
    ("mxa2a_set_option", ctypes.c_int, [_VP, ctypes.c_int, _I64]),
    ("mxa2a_get_option", ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(_I64)]),
    ("mxa2a_plan_preview", ctypes.c_int, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(_I64), ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(_I64), ctypes.c_int]),
    ("mxa2a_last_kernel_ms", ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_float)]),
    ("mxa2a_kernel_times", ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int)]),
    ("mxa2a_read_workspace", ctypes.c_int, [_VP, ctypes.c_int, _VP, ctypes.c_size_t,
                                            ctypes.POINTER(ctypes.c_size_t)]),
    ("mxa2a_l2_flush", ctypes.c_int, [_VP, ctypes.c_size_t, _VP]),
    ("mxa2a_run_noalloc", ctypes.c_int, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int, _PP, _PP, _VP,
                                         _VP, _VP, _VP]),
    ("mxa2a_destroy", None, [_VP]),
    ("mxa2a_strerror", ctypes.c_char_p, [ctypes.c_int]),
]


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Open libmxa2a.so (built by ``all_mxfp8_block_gb300.build``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise Mxa2aError(MXA2A_ERR_CUDA, f"{path} is not built (python -m all_mxfp8_block_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, res, args in _SIGS:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().mxa2a_strerror(code).decode()
    except Exception:
        return f"error {code}"


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(s) -> int:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ptr_array(xs):
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _check(rc: int, what: str):
    if rc != MXA2A_OK:
        raise Mxa2aError(rc, what)


# --- the C functions, same names ------------------------------------------------
def mxa2a_validate(R, M, kPerRank, N, commMSize, buffer_num) -> int:
    return load().mxa2a_validate(R, M, kPerRank, N, commMSize, buffer_num)


def mxa2a_plan_preview(R, M, kPerRank, N, commMSize, buffer_num, sm_count, max_pairs_fused, max_pairs_unfused,
                       options, keys) -> dict:
    """The planner's choices on the host, no device.  options: (MXA2A_OPT_*
    key, value) pairs applied in order; keys: the MXA2A_INFO_* / MXA2A_OPT_*
    keys to read.  Returns {key: value}."""
    opts = list(options)
    ok = (ctypes.c_int * max(1, len(opts)))(*[k for k, _ in opts])
    ov = (_I64 * max(1, len(opts)))(*[v for _, v in opts])
    keys = list(keys)
    ik = (ctypes.c_int * max(1, len(keys)))(*keys)
    iv = (_I64 * max(1, len(keys)))()
    _check(load().mxa2a_plan_preview(R, M, kPerRank, N, commMSize, buffer_num, sm_count, max_pairs_fused,
                                     max_pairs_unfused, ok, ov, len(opts), ik, iv, len(keys)),
           "mxa2a_plan_preview")
    return {k: int(iv[i]) for i, k in enumerate(keys)}


def plan_preview(R, M, kPerRank, N, commMSize, buffer_num, keys, options=(), sm_count=152, max_pairs_fused=76,
                 max_pairs_unfused=76) -> dict:
    """mxa2a_plan_preview with a GB300's SM and pair counts by default."""
    return mxa2a_plan_preview(R, M, kPerRank, N, commMSize, buffer_num, sm_count, max_pairs_fused,
                              max_pairs_unfused, options, keys)


def mxa2a_create(R, M, kPerRank, N, commMSize, buffer_num) -> int:
    h = load().mxa2a_create(R, M, kPerRank, N, commMSize, buffer_num)
    if not h:
        raise Mxa2aError(load().mxa2a_last_error(), "mxa2a_create")
    return h


def mxa2a_last_error() -> int:
    return load().mxa2a_last_error()


def mxa2a_validate_allgather(R, rowsPerRank, K, N, commMSize, buffer_num) -> int:
    return load().mxa2a_validate_allgather(R, rowsPerRank, K, N, commMSize, buffer_num)


def mxa2a_create_allgather(R, rowsPerRank, K, N, commMSize, buffer_num) -> int:
    h = load().mxa2a_create_allgather(R, rowsPerRank, K, N, commMSize, buffer_num)
    if not h:
        raise Mxa2aError(load().mxa2a_last_error(), "mxa2a_create_allgather")
    return h


def mxa2a_validate_reduce_scatter(R, rank, M, K, N) -> int:
    return load().mxa2a_validate_reduce_scatter(R, rank, M, K, N)


def mxa2a_create_reduce_scatter(R, rank, M, K, N) -> int:
    h = load().mxa2a_create_reduce_scatter(R, rank, M, K, N)
    if not h:
        raise Mxa2aError(load().mxa2a_last_error(), "mxa2a_create_reduce_scatter")
    return h


def mxa2a_validate_allreduce(R, rank, M, K, N) -> int:
    return load().mxa2a_validate_allreduce(R, rank, M, K, N)


def mxa2a_create_allreduce(R, rank, M, K, N) -> int:
    h = load().mxa2a_create_allreduce(R, rank, M, K, N)
    if not h:
        raise Mxa2aError(load().mxa2a_last_error(), "mxa2a_create_allreduce")
    return h


def mxa2a_run_allreduce(plan, A, A_scale, B, B_scale, recv, pub, out, stream=None) -> None:
    _check(load().mxa2a_run_allreduce(plan, _ptr(A), _ptr(A_scale), _ptr(B), _ptr(B_scale), _ptr_array(recv),
                                      _ptr(pub), _ptr(out), _stream(stream)), "mxa2a_run_allreduce")


def mxa2a_run_allreduce_unfused(plan, A, A_scale, B, B_scale, recv, pub, out, stream=None) -> None:
    _check(load().mxa2a_run_allreduce_unfused(plan, _ptr(A), _ptr(A_scale), _ptr(B), _ptr(B_scale),
                                              _ptr_array(recv), _ptr(pub), _ptr(out), _stream(stream)),
           "mxa2a_run_allreduce_unfused")


def mxa2a_run_reduce_scatter(plan, A, A_scale, B, B_scale, recv, send, out, stream=None) -> None:
    rv, sd = _ptr_array(recv), _ptr_array(send)
    _check(load().mxa2a_run_reduce_scatter(plan, _ptr(A), _ptr(A_scale), _ptr(B), _ptr(B_scale), rv, sd,
                                           _ptr(out), _stream(stream)), "mxa2a_run_reduce_scatter")


def mxa2a_run_reduce_scatter_unfused(plan, A, A_scale, B, B_scale, recv, send, out, stream=None) -> None:
    rv, sd = _ptr_array(recv), _ptr_array(send)
    _check(load().mxa2a_run_reduce_scatter_unfused(plan, _ptr(A), _ptr(A_scale), _ptr(B), _ptr(B_scale), rv, sd,
                                                   _ptr(out), _stream(stream)),
           "mxa2a_run_reduce_scatter_unfused")


def mxa2a_run(plan, A_seg, A_scale_seg, B, B_scale, C_bf16, stream=None) -> None:
    _check(load().mxa2a_run(plan, _ptr_array(A_seg), _ptr_array(A_scale_seg), _ptr(B), _ptr(B_scale),
                            _ptr(C_bf16), _stream(stream)), "mxa2a_run")


def mxa2a_run_unfused(plan, A_seg, A_scale_seg, B, B_scale, C_bf16, stream=None) -> None:
    _check(load().mxa2a_run_unfused(plan, _ptr_array(A_seg), _ptr_array(A_scale_seg), _ptr(B), _ptr(B_scale),
                                    _ptr(C_bf16), _stream(stream)), "mxa2a_run_unfused")


def mxa2a_run_direct(plan, A_seg, A_scale_seg, B, B_scale, C_bf16, stream=None) -> None:
    _check(load().mxa2a_run_direct(plan, _ptr_array(A_seg), _ptr_array(A_scale_seg), _ptr(B), _ptr(B_scale),
                                   _ptr(C_bf16), _stream(stream)), "mxa2a_run_direct")


def mxa2a_run_host(plan, A_seg, A_scale_seg, B, B_scale, C_bf16, stream=None) -> None:
    _check(load().mxa2a_run_host(plan, _ptr_array(A_seg), _ptr_array(A_scale_seg), _ptr(B), _ptr(B_scale),
                                 _ptr(C_bf16), _stream(stream)), "mxa2a_run_host")


def mxa2a_get_status(plan) -> dict:
    st = mxa2a_status()
    _check(load().mxa2a_get_status(plan, ctypes.byref(st)), "mxa2a_get_status")
    return {f: getattr(st, f) for f, _ in mxa2a_status._fields_}


def mxa2a_set_option(plan, key: int, value: int) -> None:
    _check(load().mxa2a_set_option(plan, key, int(value)), f"mxa2a_set_option({key})")


def mxa2a_get_option(plan, key: int) -> int:
    v = ctypes.c_int64()
    _check(load().mxa2a_get_option(plan, key, ctypes.byref(v)), f"mxa2a_get_option({key})")
    return v.value


def mxa2a_last_kernel_ms(plan) -> float:
    v = ctypes.c_float()
    _check(load().mxa2a_last_kernel_ms(plan, ctypes.byref(v)), "mxa2a_last_kernel_ms")
    return v.value


def mxa2a_kernel_times(plan, max_count: int) -> list:
    buf = (ctypes.c_float * max_count)()
    n = ctypes.c_int()
    _check(load().mxa2a_kernel_times(plan, buf, max_count, ctypes.byref(n)), "mxa2a_kernel_times")
    return list(buf[:n.value])


def mxa2a_read_workspace(plan, which: int):
    import numpy as np
    n = ctypes.c_size_t()
    _check(load().mxa2a_read_workspace(plan, which, None, 0, ctypes.byref(n)), "mxa2a_read_workspace")
    out = np.empty(n.value, dtype=np.uint8)
    _check(load().mxa2a_read_workspace(plan, which, out.ctypes.data, n.value, None), "mxa2a_read_workspace")
    return out


def mxa2a_l2_flush(buf, nbytes: int, stream=None) -> None:
    _check(load().mxa2a_l2_flush(_ptr(buf), nbytes, _stream(stream)), "mxa2a_l2_flush")


def mxa2a_run_noalloc(R, M, kPerRank, N, commMSize, buffer_num, A_seg, A_scale_seg, B, B_scale, C_bf16,
                      stream=None) -> None:
    """The fused path without any device allocation (static scratch inside the
    library; see include/mxa2a.h for its size limit and sharing rules)."""
    _check(load().mxa2a_run_noalloc(R, M, kPerRank, N, commMSize, buffer_num, _ptr_array(A_seg),
                                    _ptr_array(A_scale_seg), _ptr(B), _ptr(B_scale), _ptr(C_bf16),
                                    _stream(stream)), "mxa2a_run_noalloc")


def mxa2a_destroy(plan) -> None:
    if plan:
        load().mxa2a_destroy(plan)


def mxa2a_strerror(code: int) -> str:
    return strerror(code)


class Plan:
    """Owning wrapper of an ``mxa2a_plan*`` with the same calls as methods."""

    def __init__(self, R, M, kPerRank, N, commMSize, buffer_num):
        self.shape = (R, M, kPerRank, N, commMSize, buffer_num)
        self.R, self.M, self.kPerRank, self.N = R, M, kPerRank, N
        self.handle = mxa2a_create(R, M, kPerRank, N, commMSize, buffer_num)

    def run(self, A_seg, A_scale_seg, B, B_scale, C, stream=None):
        mxa2a_run(self.handle, A_seg, A_scale_seg, B, B_scale, C, stream)

    def run_unfused(self, A_seg, A_scale_seg, B, B_scale, C, stream=None):
        mxa2a_run_unfused(self.handle, A_seg, A_scale_seg, B, B_scale, C, stream)

    def run_direct(self, A_seg, A_scale_seg, B, B_scale, C, stream=None):
        mxa2a_run_direct(self.handle, A_seg, A_scale_seg, B, B_scale, C, stream)

    def run_host(self, A_seg, A_scale_seg, B, B_scale, C, stream=None):
        mxa2a_run_host(self.handle, A_seg, A_scale_seg, B, B_scale, C, stream)

    def status(self) -> dict:
        return mxa2a_get_status(self.handle)

    def set_option(self, key, value):
        mxa2a_set_option(self.handle, key, value)

    def get_option(self, key) -> int:
        return mxa2a_get_option(self.handle, key)

    def last_kernel_ms(self) -> float:
        return mxa2a_last_kernel_ms(self.handle)

    def kernel_times(self, max_count: int) -> list:
        return mxa2a_kernel_times(self.handle, max_count)

    def read_workspace(self, which):
        return mxa2a_read_workspace(self.handle, which)

    def destroy(self):
        if getattr(self, "handle", None):
            mxa2a_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class AllGatherPlan(Plan):
    """AllGather + GEMM plan (``mxa2a_create_allgather``): the run methods take
    the R row blocks ``A_blk`` / ``A_scale_blk`` in place of the segments."""

    def __init__(self, R, rowsPerRank, K, N, commMSize, buffer_num):
        self.shape = (R, rowsPerRank, K, N, commMSize, buffer_num)
        self.R, self.M, self.K, self.N = R, R * rowsPerRank, K, N
        self.handle = mxa2a_create_allgather(R, rowsPerRank, K, N, commMSize, buffer_num)


class ReduceScatterPlan(Plan):
    """GEMM + ReduceScatter plan (``mxa2a_create_reduce_scatter``) of rank
    ``rank`` of ``R``: ``run`` / ``run_unfused`` take this rank's A, B (and
    scales), the R received partial blocks ``recv`` and the R send buffers
    ``send`` (entry ``rank`` of each unused) and the output block ``out``."""

    def __init__(self, R, rank, M, K, N):
        self.shape = (R, rank, M, K, N)
        self.R, self.rank, self.M, self.K, self.N = R, rank, M, K, N
        self.rows = M // R
        self.handle = mxa2a_create_reduce_scatter(R, rank, M, K, N)

    def run(self, A, A_scale, B, B_scale, recv, send, out, stream=None):
        mxa2a_run_reduce_scatter(self.handle, A, A_scale, B, B_scale, recv, send, out, stream)

    def run_unfused(self, A, A_scale, B, B_scale, recv, send, out, stream=None):
        mxa2a_run_reduce_scatter_unfused(self.handle, A, A_scale, B, B_scale, recv, send, out, stream)

    def run_direct(self, *a, **k):
        raise Mxa2aError(MXA2A_ERR_INVALID_OPTION, "a reduce-scatter plan has run and run_unfused only")

    def run_host(self, *a, **k):
        raise Mxa2aError(MXA2A_ERR_INVALID_OPTION, "a reduce-scatter plan has run and run_unfused only")


class AllReducePlan(Plan):
    """GEMM + AllReduce (one-shot) plan (``mxa2a_create_allreduce``) of rank
    ``rank`` of ``R``: ``run`` / ``run_unfused`` take this rank's A, B (and
    scales), the R peers' published partials ``recv`` (entry ``rank`` unused),
    this rank's published partial ``pub`` and the output ``out`` (both
    [M][N] BF16)."""

    def __init__(self, R, rank, M, K, N):
        self.shape = (R, rank, M, K, N)
        self.R, self.rank, self.M, self.K, self.N = R, rank, M, K, N
        self.handle = mxa2a_create_allreduce(R, rank, M, K, N)

    def run(self, A, A_scale, B, B_scale, recv, pub, out, stream=None):
        mxa2a_run_allreduce(self.handle, A, A_scale, B, B_scale, recv, pub, out, stream)

    def run_unfused(self, A, A_scale, B, B_scale, recv, pub, out, stream=None):
        mxa2a_run_allreduce_unfused(self.handle, A, A_scale, B, B_scale, recv, pub, out, stream)

    def run_direct(self, *a, **k):
        raise Mxa2aError(MXA2A_ERR_INVALID_OPTION, "an all-reduce plan has run and run_unfused only")

    def run_host(self, *a, **k):
        raise Mxa2aError(MXA2A_ERR_INVALID_OPTION, "an all-reduce plan has run and run_unfused only")
