"""libmxa2a: fused AllToAll + MXFP8 block-scaled GEMM for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libmxa2a.so`` built from ``csrc/``;
``all_mxfp8_block_gb300.mxa2a`` is its thin ctypes binding.  Importing this
package loads nothing: the library is opened by the binding on first use and
raises if it has not been built.
"""
__all__ = ["inputs", "mxa2a"]
