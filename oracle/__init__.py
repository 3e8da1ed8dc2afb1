"""CPU oracle of the asymmetric group-wise W4A16 linear layer (numpy front end to oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()`` and by the
``cpu_baseline`` / reference leg of ``bench.py``.  The product library never imports it, and
it imports nothing from the product.  All arithmetic is in oracle.c (IEEE double); this module
only marshals numpy arrays.

Layer definition (see oracle.c for the page citations): with q and z 4-bit codes and s fp16,
``W[k, n] = (q[k, n] - z[k // g, n]) * s[k // g, n]`` and ``y = x @ W``.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, invariants, brute force, exhaustive fp16 checks).
The only unpinned reading is the tail block of the CPU ``[N/64][K][32 bytes]`` layout when N is
not a multiple of 64 (padded with code 0 here): "parity unpinned" for that tail.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        sig = {
            "oracle_num_threads": ([], I),
            "oracle_half_to_double": ([ctypes.c_uint16], ctypes.c_double),
            "oracle_double_to_half": ([ctypes.c_double], ctypes.c_uint16),
            "oracle_double_to_half_array": ([P, I64, P], None),
            "oracle_half_to_double_array": ([P, I64, P], None),
            "oracle_awq_unpack": ([P, I, I, P], None),
            "oracle_awq_pack": ([P, I, I, P], None),
            "oracle_dequant_codes_f64": ([P, P, P, I, I, I, P], None),
            "oracle_dequant_awq_f64": ([P, P, P, I, I, I, P], I),
            "oracle_dequant_awq_f16": ([P, P, P, I, I, I, P], I),
            "oracle_gemm_f64": ([P, I, I, P, I, P], None),
            "oracle_linear": ([P, I, I, P, P, P, I, I, P, P], I),
            "oracle_linear_sampled": ([P, I, I, P, P, P, I, I, P, P, I64, P], None),
            "oracle_awq_to_standard": ([P, P, I, I, I, P, P], None),
            "oracle_dequant_standard_f64": ([P, P, P, I, I, I, P], None),
            "oracle_int4pack_cpu_chunk": ([P, I, I, I, I, P], None),
            "oracle_int4pack_cpu": ([P, I, I, P], None),
            "oracle_int4unpack_cpu": ([P, I, I, P], None),
            "oracle_embed_gather": ([P, P, P, I, I, I, P, I, P], I),
            "oracle_bf16_to_double": ([ctypes.c_uint16], ctypes.c_double),
            "oracle_double_to_bf16": ([ctypes.c_double], ctypes.c_uint16),
            "oracle_double_to_bf16_array": ([P, I64, P], None),
            "oracle_dequant_awq_bf16_f64": ([P, P, P, I, I, I, P], I),
            "oracle_dequant_awq_bf16": ([P, P, P, I, I, I, P], I),
            "oracle_linear_bf16": ([P, I, I, P, P, P, I, I, P, P], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _c(a, dtype):
    """C-contiguous array of exactly ``dtype`` (no value conversion for integer bit patterns)."""
    a = np.asarray(a)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iuf" and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return np.ascontiguousarray(a)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads():
    return lib().oracle_num_threads()


# ------------------------------------------------------------------ binary16

def half_bits_to_double(h):
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float64)
    lib().oracle_half_to_double_array(_p(h), h.size, _p(out))
    return out


def double_to_half_bits(v):
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_double_to_half_array(_p(v), v.size, _p(out))
    return out


# ------------------------------------------------------------------ AWQ packing

def awq_unpack(packed, N):
    packed = _c(packed, np.int32)
    rows = packed.shape[0]
    assert packed.shape == (rows, N // 8)
    codes = np.empty((rows, N), np.uint8)
    lib().oracle_awq_unpack(_p(packed), rows, N, _p(codes))
    return codes


def awq_pack(codes):
    codes = _c(codes, np.uint8)
    rows, N = codes.shape
    packed = np.empty((rows, N // 8), np.int32)
    lib().oracle_awq_pack(_p(codes), rows, N, _p(packed))
    return packed


# ------------------------------------------------------------------ dequantization

def dequant_codes_f64(q, z, scales_bits, g):
    q = _c(q, np.uint8)
    z = _c(z, np.uint8)
    s = _c(scales_bits, np.uint16)
    K, N = q.shape
    W = np.empty((K, N), np.float64)
    lib().oracle_dequant_codes_f64(_p(q), _p(z), _p(s), K, N, g, _p(W))
    return W


def dequant_f64(qweight, qzeros, scales_bits, K, N, g):
    qw, qz, s = _c(qweight, np.int32), _c(qzeros, np.int32), _c(scales_bits, np.uint16)
    W = np.empty((K, N), np.float64)
    if lib().oracle_dequant_awq_f64(_p(qw), _p(qz), _p(s), K, N, g, _p(W)):
        raise MemoryError("oracle_dequant_awq_f64")
    return W


def dequant_f16_bits(qweight, qzeros, scales_bits, K, N, g):
    qw, qz, s = _c(qweight, np.int32), _c(qzeros, np.int32), _c(scales_bits, np.uint16)
    W = np.empty((K, N), np.uint16)
    if lib().oracle_dequant_awq_f16(_p(qw), _p(qz), _p(s), K, N, g, _p(W)):
        raise MemoryError("oracle_dequant_awq_f16")
    return W


def embed_gather(qweight, qzeros, scales_bits, K, N, g, ids):
    """fp16 bits [T, K]: row t is column ids[t] of the dequantized W (zeros for ids outside
    [0, N)); also returns the number of such ids."""
    qw, qz, s = _c(qweight, np.int32), _c(qzeros, np.int32), _c(scales_bits, np.uint16)
    ids = _c(ids, np.int32)
    out = np.empty((len(ids), K), np.uint16)
    bad = lib().oracle_embed_gather(_p(qw), _p(qz), _p(s), K, N, g, _p(ids), len(ids), _p(out))
    return out, bad


# ------------------------------------------------------------------ the linear layer

def gemm_f64(x_bits, W):
    x = _c(x_bits, np.uint16)
    W = _c(W, np.float64)
    M, K = x.shape
    K2, N = W.shape
    assert K == K2
    y = np.empty((M, N), np.float64)
    lib().oracle_gemm_f64(_p(x), M, K, _p(W), N, _p(y))
    return y


def linear(x_bits, qweight, qzeros, scales_bits, K, N, g):
    """Returns (y in double, y rounded to fp16 bits)."""
    x = _c(x_bits, np.uint16)
    M = x.shape[0]
    qw, qz, s = _c(qweight, np.int32), _c(qzeros, np.int32), _c(scales_bits, np.uint16)
    y64 = np.empty((M, N), np.float64)
    y16 = np.empty((M, N), np.uint16)
    if lib().oracle_linear(_p(x), M, K, _p(qw), _p(qz), _p(s), N, g, _p(y64), _p(y16)):
        raise MemoryError("oracle_linear")
    return y64, y16


def linear_sampled(x_bits, qweight, qzeros, scales_bits, K, N, g, m_idx, n_idx):
    x = _c(x_bits, np.uint16)
    M = x.shape[0]
    qw, qz, s = _c(qweight, np.int32), _c(qzeros, np.int32), _c(scales_bits, np.uint16)
    mi = _c(m_idx, np.int64)
    ni = _c(n_idx, np.int64)
    assert mi.shape == ni.shape
    out = np.empty(mi.shape, np.float64)
    lib().oracle_linear_sampled(_p(x), M, K, _p(qw), _p(qz), _p(s), N, g, _p(mi), _p(ni), mi.size, _p(out))
    return out


# ------------------------------------------------------------------ other layouts

def awq_to_standard(qweight, qzeros, K, N, g):
    qw, qz = _c(qweight, np.int32), _c(qzeros, np.int32)
    qw_std = np.empty((K // 8, N), np.int32)
    qz_std = np.empty((K // g, N // 8), np.int32)
    lib().oracle_awq_to_standard(_p(qw), _p(qz), K, N, g, _p(qw_std), _p(qz_std))
    return qw_std, qz_std


def dequant_standard_f64(qweight_std, qzeros_std, scales_bits, K, N, g):
    qw, qz, s = _c(qweight_std, np.int32), _c(qzeros_std, np.int32), _c(scales_bits, np.uint16)
    W = np.empty((K, N), np.float64)
    lib().oracle_dequant_standard_f64(_p(qw), _p(qz), _p(s), K, N, g, _p(W))
    return W


def int4pack_cpu(q, n0=None, n1=None, out=None):
    """The CPU kernel's [ceil(N/64)][K][32 bytes] layout; optionally only n-blocks in [n0, n1)."""
    q = _c(q, np.uint8)
    K, N = q.shape
    nb = (N + 63) // 64
    if out is None:
        out = np.zeros((nb, K, 32), np.uint8)
    if n0 is None:
        lib().oracle_int4pack_cpu(_p(q), K, N, _p(out))
    else:
        lib().oracle_int4pack_cpu_chunk(_p(q), K, N, n0, n1, _p(out))
    return out


def int4unpack_cpu(packed, K, N):
    packed = _c(packed, np.uint8)
    q = np.empty((K, N), np.uint8)
    lib().oracle_int4unpack_cpu(_p(packed), K, N, _p(q))
    return q


# ------------------------------------------------------------------ the bf16 layer

def bf16_bits_to_double(b):
    b = _c(b, np.uint16)
    f = np.vectorize(lib().oracle_bf16_to_double, otypes=[np.float64])
    return f(b) if b.size else np.empty(b.shape, np.float64)


def double_to_bf16_bits(v):
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_double_to_bf16_array(_p(v), v.size, _p(out))
    return out


def dequant_bf16_bits(qweight, qzeros, scales_bits, K, N, g):
    qw, qz, s = _c(qweight, np.int32), _c(qzeros, np.int32), _c(scales_bits, np.uint16)
    W = np.empty((K, N), np.uint16)
    if lib().oracle_dequant_awq_bf16(_p(qw), _p(qz), _p(s), K, N, g, _p(W)):
        raise MemoryError("oracle_dequant_awq_bf16")
    return W


def linear_bf16(x_bits, qweight, qzeros, scales_bits, K, N, g):
    """bf16 layer: returns (y in double, y rounded to bfloat16 bits)."""
    x = _c(x_bits, np.uint16)
    M = x.shape[0]
    qw, qz, s = _c(qweight, np.int32), _c(qzeros, np.int32), _c(scales_bits, np.uint16)
    y64 = np.empty((M, N), np.float64)
    yb = np.empty((M, N), np.uint16)
    if lib().oracle_linear_bf16(_p(x), M, K, _p(qw), _p(qz), _p(s), N, g, _p(y64), _p(yb)):
        raise MemoryError("oracle_linear_bf16")
    return y64, yb
