"""The C-ABI library loads, exports every entry point include/w4a16.h declares, and rejects bad
arguments on the host (these calls return before any CUDA call, so no GPU is needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import __graft_entry__
from w4a16_group_wise_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return binding.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "w4a16_gemm" in names and "w4a16_repack" in names and "w4a16_dequant" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) <= set(binding.SIGNATURES)


@pytest.mark.parametrize("path", [binding.LIB_PATH, binding.BOUNDS_LIB_PATH])
def test_exports_nothing_undeclared(L, path):
    """The normal library and its bounds-checked build export the same declared entry points."""
    out = os.popen("nm -D --defined-only %s" % path).read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and "w4a16" in l}
    assert exported == set(_declared())


def test_which_build(L):
    assert L.w4a16_bounds_checked() == 0
    with binding.bounds_checked_library() as B:
        assert B.w4a16_bounds_checked() == 1 and binding.lib() is B
    assert binding.lib() is L


def test_layout_version_and_sizes(L):
    assert L.w4a16_layout_version() == 1
    # 256-byte header + ceil(N/64) * ceil(K/128) chunks of 4096 + (128/g) * 160 bytes
    assert L.w4a16_packed_bytes(2048, 13312, 128) == 256 + 208 * 16 * 4256
    assert L.w4a16_packed_bytes(6656, 80, 32) == 256 + 2 * 52 * (4096 + 4 * 160)
    assert L.w4a16_packed_bytes(96, 8, 32) == 256 + 1 * 1 * 4736
    assert L.w4a16_packed_bytes(2048, 2048, 100) == 0
    assert L.w4a16_packed_bytes(2048, 2044, 128) == 0
    assert L.w4a16_packed_bytes(2000, 2048, 128) == 0
    assert L.w4a16_packed_bytes(0, 2048, 128) == 0
    assert L.w4a16_workspace_bytes(1, 2048, 2048, 128) == 0


P = ctypes.c_void_p(0x10000)       # aligned, never dereferenced: every case below fails first
P_ODD = ctypes.c_void_p(0x10008)
NUL = ctypes.c_void_p(0)


@pytest.mark.parametrize("args,status", [
    ((P, P, 1, 2048, 2048, 100, P, NUL, 0, NUL), binding.ERR_UNSUPPORTED),   # g
    ((P, P, 1, 2044, 2048, 128, P, NUL, 0, NUL), binding.ERR_UNSUPPORTED),   # N % 8
    ((P, P, 1, 2048, 2000, 128, P, NUL, 0, NUL), binding.ERR_UNSUPPORTED),   # K % g
    ((P, P, -1, 2048, 2048, 128, P, NUL, 0, NUL), binding.ERR_INVALID),      # M < 0
    ((P, P, 1, 0, 2048, 128, P, NUL, 0, NUL), binding.ERR_INVALID),          # N = 0
    ((NUL, P, 1, 2048, 2048, 128, P, NUL, 0, NUL), binding.ERR_INVALID),     # x null
    ((P, NUL, 1, 2048, 2048, 128, P, NUL, 0, NUL), binding.ERR_INVALID),     # packed null
    ((P, P, 1, 2048, 2048, 128, NUL, NUL, 0, NUL), binding.ERR_INVALID),     # y null
    ((P_ODD, P, 1, 2048, 2048, 128, P, NUL, 0, NUL), binding.ERR_MISALIGNED),
    ((P, P, 1, 2048, 2048, 128, P_ODD, NUL, 0, NUL), binding.ERR_MISALIGNED),
    ((P, P, 0, 2048, 2048, 128, NUL, NUL, 0, NUL), binding.OK),              # M = 0: no-op
])
def test_gemm_host_validation(L, args, status):
    assert L.w4a16_gemm(*args) == status


def test_repack_and_dequant_host_validation(L):
    assert L.w4a16_repack(P, P, P, 2048, 2048, 96, P, NUL) == binding.ERR_UNSUPPORTED
    assert L.w4a16_repack(NUL, P, P, 2048, 2048, 128, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_repack(P, P, P, 2048, 2048, 128, P_ODD, NUL) == binding.ERR_MISALIGNED
    assert L.w4a16_dequant(P, 2048, 2048, 64, NUL, NUL) == binding.ERR_INVALID
    assert L.w4a16_dequant(P, 2048, 2050, 64, P, NUL) == binding.ERR_UNSUPPORTED
    assert L.w4a16_dequant(P_ODD, 2048, 2048, 64, P, NUL) == binding.ERR_MISALIGNED


@pytest.mark.parametrize("n0,n1", [(32, 128), (0, 100), (128, 64), (0, 0), (-64, 64), (0, 2112)])
def test_repack_chunk_rejects_bad_ranges(L, n0, n1):
    # N = 2048: n0 must be a multiple of 64, n1 a multiple of 64 or N, 0 <= n0 < n1 <= N
    st = L.w4a16_repack_chunk(P, 256, P, 256, P, 2048, 2048, 2048, 128, n0, n1, P, NUL)
    assert st == binding.ERR_INVALID


def test_repack_chunk_rejects_short_strides(L):
    assert L.w4a16_repack_chunk(P, 7, P, 8, P, 64, 2048, 2048, 128, 0, 64, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_repack_chunk(P, 8, P, 8, P, 63, 2048, 2048, 128, 0, 64, P, NUL) == binding.ERR_INVALID


def test_status_strings(L):
    for s in range(-6, 1):
        assert binding.status_string(s) and "unknown" not in binding.status_string(s)
    assert "unknown" in binding.status_string(-99)


def test_set_option_validation(L):
    assert L.w4a16_set_option(1, 0) == binding.OK
    assert L.w4a16_set_option(1, 1) == binding.OK
    assert L.w4a16_set_option(1, 0) == binding.OK
    assert L.w4a16_set_option(1, 7) == binding.ERR_INVALID
    assert L.w4a16_set_option(99, 0) == binding.ERR_INVALID


def test_embed_host_validation(L):
    # every case is rejected before any launch (the pointers are never dereferenced)
    P4 = ctypes.c_void_p(0x10004)                                                     # 4- but not 16-byte aligned
    assert L.w4a16_embed(P, 4, P, 2048, 2048, 100, P, NUL) == binding.ERR_UNSUPPORTED  # g
    assert L.w4a16_embed(P, -1, P, 2048, 2048, 128, P, NUL) == binding.ERR_INVALID     # T < 0
    assert L.w4a16_embed(NUL, 4, P, 2048, 2048, 128, P, NUL) == binding.ERR_INVALID    # ids null
    assert L.w4a16_embed(P, 4, P, 2048, 2048, 128, NUL, NUL) == binding.ERR_INVALID    # out null
    assert L.w4a16_embed(P, 4, P, 2048, 2048, 128, P4, NUL) == binding.ERR_MISALIGNED  # out
    assert L.w4a16_embed(ctypes.c_void_p(0x10002), 4, P, 2048, 2048, 128, P, NUL) == binding.ERR_MISALIGNED
    assert L.w4a16_embed(NUL, 0, NUL, 2048, 2048, 128, NUL, NUL) == binding.OK          # T = 0: no-op


def test_per_channel_group_sizes(L):
    """One group over all of K (g == K or g == -1) is stored with the largest of 128, 64, 32
    dividing K; K % 32 != 0 is unsupported; other g values are rejected."""
    assert L.w4a16_packed_bytes(2048, 3072, -1) == L.w4a16_packed_bytes(2048, 3072, 128)
    assert L.w4a16_packed_bytes(2048, 3072, 2048) == L.w4a16_packed_bytes(2048, 3072, 128)
    assert L.w4a16_packed_bytes(192, 136, 192) == L.w4a16_packed_bytes(192, 136, 64)
    assert L.w4a16_packed_bytes(160, 80, -1) == L.w4a16_packed_bytes(160, 80, 32)
    assert L.w4a16_packed_bytes(200, 80, -1) == 0                     # K % 32 != 0
    assert L.w4a16_packed_bytes(2048, 3072, 256) == 0                 # neither 32/64/128 nor K
    assert L.w4a16_gemm(P, P, 1, 3072, 2048, -2, P, NUL, 0, NUL) == binding.ERR_INVALID
    assert L.w4a16_gemm(P, P, 1, 80, 200, -1, P, NUL, 0, NUL) == binding.ERR_UNSUPPORTED


def test_awq_to_standard_host_validation(L):
    # every case is rejected before any launch (the pointers are never dereferenced)
    P2 = ctypes.c_void_p(0x10002)
    assert L.w4a16_awq_to_standard(P, P, 2048, 3072, 100, P, P, NUL) == binding.ERR_UNSUPPORTED
    assert L.w4a16_awq_to_standard(NUL, P, 2048, 3072, 128, P, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_awq_to_standard(P, P, 2048, 3072, 128, P, NUL, NUL) == binding.ERR_INVALID
    assert L.w4a16_awq_to_standard(P, P, 2048, 3072, 128, P2, P, NUL) == binding.ERR_MISALIGNED
    assert L.w4a16_awq_to_standard(P, P2, 2048, 3072, 128, P, P, NUL) == binding.ERR_MISALIGNED
    assert L.w4a16_awq_to_standard(P, P, 2048, 3072, 128, ctypes.c_void_p(0x10004), P, NUL) == binding.ERR_MISALIGNED


def test_bf16_entry_points_host_validation(L):
    # the bf16 entry points validate exactly as their fp16 counterparts (rejected before any launch)
    assert L.w4a16_gemm_bf16(P, P, 1, 2048, 2048, 100, P, NUL, 0, NUL) == binding.ERR_UNSUPPORTED
    assert L.w4a16_gemm_bf16(P, P, -1, 2048, 2048, 128, P, NUL, 0, NUL) == binding.ERR_INVALID
    assert L.w4a16_gemm_bf16(NUL, P, 1, 2048, 2048, 128, P, NUL, 0, NUL) == binding.ERR_INVALID
    assert L.w4a16_gemm_bf16(P_ODD, P, 1, 2048, 2048, 128, P, NUL, 0, NUL) == binding.ERR_MISALIGNED
    assert L.w4a16_gemm_bf16(P, P, 0, 2048, 2048, 128, NUL, NUL, 0, NUL) == binding.OK
    assert L.w4a16_repack_bf16(P, P, P, 2048, 2048, 96, P, NUL) == binding.ERR_UNSUPPORTED
    assert L.w4a16_repack_bf16(P, P, P, 2048, 2048, 128, P_ODD, NUL) == binding.ERR_MISALIGNED
    assert L.w4a16_repack_chunk_bf16(P, 256, P, 256, P, 2048, 2048, 2048, 128, 32, 128, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_repack_chunk_bf16(P, 7, P, 8, P, 64, 2048, 2048, 128, 0, 64, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_dequant_bf16(P, 2048, 2048, 64, NUL, NUL) == binding.ERR_INVALID
    assert L.w4a16_dequant_bf16(P_ODD, 2048, 2048, 64, P, NUL) == binding.ERR_MISALIGNED
    assert L.w4a16_embed_bf16(P, -1, P, 2048, 2048, 128, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_embed_bf16(NUL, 0, NUL, 2048, 2048, 128, NUL, NUL) == binding.OK


def test_bf16_inputs_are_rounded_draws():
    """The bf16 input recipe: the same draws as fp16, rounded to bfloat16 (bits as uint16)."""
    from w4a16_group_wise_gb300 import inputs
    x16 = inputs.make_x(3, 256, seed=4)
    xb = inputs.make_x(3, 256, seed=4, dtype="bf16")
    assert xb.dtype == np.uint16 and xb.shape == (3, 256)
    wide = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # both round the same normal draws: they agree to bf16's precision
    assert np.all(np.abs(wide - x16.astype(np.float64)) <= 2.0 ** -8 * np.abs(x16.astype(np.float64)) + 1e-3)
    h = inputs.make_weights(256, 64, 128, seed=1, dtype="bf16")
    hf = inputs.make_weights(256, 64, 128, seed=1)
    assert np.array_equal(h["qweight"], hf["qweight"]) and np.array_equal(h["qzeros"], hf["qzeros"])
    s = (h["scales"].astype(np.uint32) << 16).view(np.float32)
    assert np.all((s >= 0.002 * (1 - 2 ** -8)) & (s <= 0.02 * (1 + 2 ** -8)))


def test_selftest_wait_timeout_host_validation(L):
    # rejected before any launch (the pointer is never dereferenced)
    assert L.w4a16_selftest_wait_timeout(0, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_selftest_wait_timeout(-5, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_selftest_wait_timeout(200_000_000, P, NUL) == binding.ERR_INVALID
    assert L.w4a16_selftest_wait_timeout(1_000_000, NUL, NUL) == binding.ERR_INVALID
    assert L.w4a16_selftest_wait_timeout(1_000_000, ctypes.c_void_p(0x10002), NUL) == binding.ERR_MISALIGNED
