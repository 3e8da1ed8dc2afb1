"""GB300 (sm_103a) asymmetric group-wise W4A16 linear layer.

    y = x . W,   W[k, n] = (q[k, n] - z[k // g, n]) * s[k // g, n]

The compute is a C-ABI CUDA library (include/w4a16.h, csrc/); ``binding`` marshals torch
tensors into it.  ``inputs`` draws the seeded synthetic tensors used by tests and benchmarks.
"""
from .binding import (W4A16Error, awq_to_standard, bounds_checked, bounds_checked_library, dequant, embed,  # noqa: F401
                      gemm, gemm_noalloc, last_device_error, layout_version, packed_bytes, repack, repack_chunk,
                      selftest_bounds, selftest_wait_timeout, set_option, status_string, workspace_bytes)
from .shard import ColumnParallelLinear, column_slices, repack_slice  # noqa: F401
