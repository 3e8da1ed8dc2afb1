"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU needed).

Each test names the fact it pins.  They are chosen so that a plausible slip anywhere in the
oracle fails one of them: a wrong AWQ slot order (closed-form words), an arithmetic instead of
a logical shift (words with the top bit set), a wrong zero sign or offset (q == z, z = 8), a
wrong group index (per-group patterns, exact brute force), a transposed operand (M = 1 against
a library mat-vec on non-square shapes), a rounding slip (exhaustive binary16 checks).
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from w4a16_group_wise_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
AWQ_ORDER = [0, 2, 4, 6, 1, 3, 5, 7]   # slot j -> column offset (the AWQ format's interleave)


# ----------------------------------------------------------------------------- binary16

def _finite_half_bits():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (h >> 10) & 0x1F
    return h[exp != 31]


def test_half_to_double_matches_numpy_for_every_pattern():
    h = _finite_half_bits()
    ours = oracle.half_bits_to_double(h)
    ref = h.view(np.float16).astype(np.float64)      # library conversion (exact widening)
    assert np.array_equal(ours, ref)
    assert np.array_equal(np.signbit(ours), np.signbit(ref))


def test_half_round_trip_every_pattern():
    h = _finite_half_bits()
    assert np.array_equal(oracle.double_to_half_bits(oracle.half_bits_to_double(h)), h)
    inf = np.array([0x7C00, 0xFC00], np.uint16)
    assert np.array_equal(oracle.double_to_half_bits(oracle.half_bits_to_double(inf)), inf)


def test_half_rounding_at_every_midpoint_is_to_even():
    pos = np.arange(0, 0x7C00, dtype=np.uint16)            # +0 .. max finite
    v = oracle.half_bits_to_double(pos)
    mids = (v[:-1] + v[1:]) / 2                             # exact in double
    got = oracle.double_to_half_bits(mids)
    lo, hi = pos[:-1], pos[1:]
    expect = np.where(lo % 2 == 0, lo, hi)                  # the even significand wins
    assert np.array_equal(got, expect)
    # just off the midpoint goes to the nearer neighbour
    eps = (v[1:] - v[:-1]) / 1024
    assert np.array_equal(oracle.double_to_half_bits(mids - eps), lo)
    assert np.array_equal(oracle.double_to_half_bits(mids + eps), hi)
    # negatives mirror
    assert np.array_equal(oracle.double_to_half_bits(-mids), expect | 0x8000)
    # numpy's direct double -> half conversion agrees on all of them
    assert np.array_equal(mids.astype(np.float16).view(np.uint16), expect)


def test_half_rounding_is_nearest_by_brute_force():
    grid_bits = np.arange(0, 0x7C00, dtype=np.uint16)
    grid = oracle.half_bits_to_double(grid_bits)
    rng = np.random.default_rng(1)
    v = np.concatenate([
        np.exp(rng.uniform(np.log(1e-9), np.log(65000.0), 20000)),
        rng.uniform(0, 1e-4, 5000),
        rng.uniform(60000, 65504, 2000),
    ])
    got = oracle.double_to_half_bits(v)
    idx = np.searchsorted(grid, v)
    idx = np.clip(idx, 1, len(grid) - 1)
    below, above = grid[idx - 1], grid[idx]
    nearest = np.where(v - below < above - v, idx - 1, idx)
    tie = (v - below) == (above - v)
    nearest = np.where(tie, np.where((idx - 1) % 2 == 0, idx - 1, idx), nearest)
    assert np.array_equal(got, grid_bits[nearest])


def test_half_overflow_and_underflow_edges():
    f = oracle.double_to_half_bits
    assert f(np.array([65504.0]))[0] == 0x7BFF
    assert f(np.array([65519.99]))[0] == 0x7BFF
    assert f(np.array([65520.0]))[0] == 0x7C00              # tie with 2^16 goes to even -> inf
    assert f(np.array([1e6]))[0] == 0x7C00
    assert f(np.array([2.0 ** -25]))[0] == 0x0000           # tie between 0 and 2^-24 -> 0
    assert f(np.array([2.0 ** -25 * 1.0000001]))[0] == 0x0001
    assert f(np.array([3 * 2.0 ** -25]))[0] == 0x0002       # tie between 1 and 2 ulps -> 2
    assert f(np.array([-0.0]))[0] == 0x8000
    assert f(np.array([2.0 ** -14 - 2.0 ** -26]))[0] == 0x0400   # rounds up into the normals


# ----------------------------------------------------------------------------- AWQ packing

def test_awq_word_closed_form():
    """q[k, n] = n mod 8 puts code ORD[j] in slot j: every word is 0x75316420."""
    K, N = 16, 64
    q = np.tile(np.arange(N) % 8, (K, 1)).astype(np.uint8)
    words = oracle.awq_pack(q).view(np.uint32)
    assert np.all(words == 0x75316420)
    assert np.array_equal(oracle.awq_unpack(np.full((K, N // 8), 0x75316420, np.uint32), N), q)


def test_awq_each_slot_each_value():
    """All 16 values in all 8 slots: exactly column 8c + ORD[j] of row r changes."""
    N = 16
    for j in range(8):
        for v in range(16):
            w = np.zeros((2, N // 8), np.uint32)
            w[1, 1] = np.uint32(v << (4 * j))
            codes = oracle.awq_unpack(w, N)
            expect = np.zeros((2, N), np.uint8)
            expect[1, 8 + AWQ_ORDER[j]] = v
            assert np.array_equal(codes, expect), (j, v)


def test_awq_top_nibble_of_negative_words():
    """Words are read as unsigned: int32 words with the top bit set keep their top nibble."""
    w = np.array([[np.int32(-1), np.int32(np.uint32(0xF0000000).view(np.int32))]], np.int32)
    codes = oracle.awq_unpack(w, 16)
    assert np.all(codes[0, :8] == 15)
    assert codes[0, 8 + 7] == 15 and np.all(np.delete(codes[0, 8:], 7) == 0)


def test_awq_round_trip_random():
    rng = np.random.default_rng(2)
    w = rng.integers(0, 2**32, size=(37, 24), dtype=np.uint32).view(np.int32)
    codes = oracle.awq_unpack(w, 192)
    assert codes.max() <= 15
    assert np.array_equal(oracle.awq_pack(codes), w)


def test_awq_packs_along_output_dimension():
    """qweight is [K, N/8] (packed_dim = 1): a word of row k only carries row k's codes."""
    rng = np.random.default_rng(3)
    K, N = 8, 32
    w = rng.integers(0, 2**32, size=(K, N // 8), dtype=np.uint32).view(np.int32)
    base = oracle.awq_unpack(w, N)
    w2 = w.copy()
    w2[5, 2] ^= np.int32(0x0F)                   # flip slot 0 of row 5, word 2
    changed = np.argwhere(oracle.awq_unpack(w2, N) != base)
    assert changed.tolist() == [[5, 16 + AWQ_ORDER[0]]]


# ----------------------------------------------------------------------------- dequant / GEMM

def _layer(K, N, g, seed=0, **kw):
    L = inputs.make_weights(K, N, g, seed=seed, **kw)
    return L["qweight"], L["qzeros"], L["scales"].view(np.uint16)


def test_q_equal_z_gives_exact_zero():
    K, N, g = 256, 64, 128
    _, qz, s = _layer(K, N, g)
    qw = np.repeat(qz, g, axis=0)               # every code equals its group's zero
    W = oracle.dequant_f64(qw, qz, s, K, N, g)
    assert np.all(W == 0) and not np.any(np.signbit(W))
    x = inputs.make_x(3, K).view(np.uint16)
    y64, y16 = oracle.linear(x, qw, qz, s, K, N, g)
    assert np.all(y64 == 0) and np.all(y16 == 0)


def test_symmetric_grid_unit_scale_is_integer_matmul():
    """z = 8, s = 1: W = q - 8 and y is the textbook integer product."""
    K, N, g = 384, 48, 128
    qw, qz, _ = _layer(K, N, g, zeros="sym8")
    s = np.full((K // g, N), 0x3C00, np.uint16)           # 1.0
    q = oracle.awq_unpack(qw, N).astype(np.int64)
    W = oracle.dequant_f64(qw, qz, s, K, N, g)
    assert np.array_equal(W, (q - 8).astype(np.float64))
    rng = np.random.default_rng(4)
    xi = rng.integers(-3, 4, size=(5, K))
    y64, _ = oracle.linear(xi.astype(np.float16).view(np.uint16), qw, qz, s, K, N, g)
    assert np.array_equal(y64, (xi @ (q - 8)).astype(np.float64))


def test_group_index_is_floor_k_over_g():
    """Scale of group G = 2^-G and zero 0: W[k, n] = q * 2^-(k // g) exactly."""
    K, N, g = 512, 16, 64
    qw, _, _ = _layer(K, N, g)
    qz = np.zeros((K // g, N // 8), np.int32)
    s = np.stack([np.full(N, np.float16(2.0 ** -G)) for G in range(K // g)]).view(np.uint16)
    q = oracle.awq_unpack(qw, N).astype(np.float64)
    W = oracle.dequant_f64(qw, qz, s, K, N, g)
    assert np.array_equal(W, q * (2.0 ** -(np.arange(K) // g))[:, None])


def test_bit_exact_case_is_order_independent():
    """x in {-2..2}, s = 2^-8: every product and partial sum is exact, so y is exact."""
    K, N, g = 2048, 64, 128
    qw, qz, _ = _layer(K, N, g)
    s = np.full((K // g, N), np.float16(2.0 ** -8)).view(np.uint16)
    rng = np.random.default_rng(5)
    xi = rng.integers(-2, 3, size=(4, K))
    q = oracle.awq_unpack(qw, N).astype(np.int64)
    z = np.repeat(oracle.awq_unpack(qz, N).astype(np.int64), g, axis=0)
    exact = (xi @ (q - z)).astype(np.float64) * 2.0 ** -8
    y64, y16 = oracle.linear(xi.astype(np.float16).view(np.uint16), qw, qz, s, K, N, g)
    assert np.array_equal(y64, exact)
    assert np.array_equal(y16, exact.astype(np.float16).view(np.uint16))


def test_m1_is_matvec_against_library():
    K, N, g = 640, 200, 128
    qw, qz, s = _layer(K, N, g, seed=7)
    x = inputs.make_x(1, K, seed=7)
    W = oracle.dequant_f64(qw, qz, s, K, N, g)
    y64, _ = oracle.linear(x.view(np.uint16), qw, qz, s, K, N, g)
    ref = np.dot(W.T, x[0].astype(np.float64))             # library mat-vec
    assert np.allclose(y64[0], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def _exact_linear(x, qweight, qzeros, scales_bits, K, N, g):
    """Exact rational y from the AWQ words, by brute force (tiny sizes only)."""
    sv = scales_bits.view(np.float16).astype(np.float64)
    xv = x.astype(np.float64)
    out = []
    for m in range(x.shape[0]):
        row = []
        for n in range(N):
            c, j = n // 8, AWQ_ORDER.index(n % 8)
            acc = Fraction(0)
            for k in range(K):
                qc = (int(qweight[k, c]) & 0xFFFFFFFF) >> (4 * j) & 0xF
                zc = (int(qzeros[k // g, c]) & 0xFFFFFFFF) >> (4 * j) & 0xF
                acc += Fraction(xv[m, k]) * (qc - zc) * Fraction(sv[k // g, n])
            row.append(acc)
        out.append(row)
    return out


@pytest.mark.parametrize("K,N,g", [(8, 8, 8), (16, 8, 8), (32, 16, 16), (64, 32, 32),
                                   (64, 64, 16), (32, 64, 32), (64, 16, 64), (16, 32, 8)])
def test_brute_force_tiny_exact(K, N, g):
    qw, qz, s = _layer(K, N, g, seed=K * 131 + N)
    x = inputs.make_x(2, K, seed=K + N)
    exact = _exact_linear(x, qw, qz, s, K, N, g)
    y64, y16 = oracle.linear(x.view(np.uint16), qw, qz, s, K, N, g)
    for m in range(2):
        for n in range(N):
            e = exact[m][n]
            # a double sum of K exact products: error at most K * 2^-53 * sum|terms|
            assert abs(Fraction(y64[m, n]) - e) <= Fraction(K, 2**52) * (abs(e) + 64)
    # and the dequantized weights are exact
    W = oracle.dequant_f64(qw, qz, s, K, N, g)
    q = oracle.awq_unpack(qw, N).astype(np.float64)
    z = np.repeat(oracle.awq_unpack(qz, N).astype(np.float64), g, axis=0)
    assert np.array_equal(W, (q - z) * np.repeat(s.view(np.float16).astype(np.float64), g, axis=0))


def test_dequant_f16_is_single_rounding():
    K, N, g = 512, 128, 128
    qw, qz, s = _layer(K, N, g, scale_dist="loguniform", scale_lo=1e-4, scale_hi=0.1)
    W64 = oracle.dequant_f64(qw, qz, s, K, N, g)
    W16 = oracle.dequant_f16_bits(qw, qz, s, K, N, g)
    assert np.array_equal(W16, W64.astype(np.float16).view(np.uint16))   # library rounding
    # |q - z| <= 15 times an 11-bit significand is exact in float32 too
    assert np.array_equal(W64.astype(np.float32).astype(np.float64), W64)


def test_sampled_outputs_equal_full_product():
    K, N, g, M = 768, 136, 64, 3
    qw, qz, s = _layer(K, N, g, seed=9)
    x = inputs.make_x(M, K, seed=9).view(np.uint16)
    y64, _ = oracle.linear(x, qw, qz, s, K, N, g)
    rng = np.random.default_rng(6)
    mi = rng.integers(0, M, 300)
    ni = rng.integers(0, N, 300)
    ys = oracle.linear_sampled(x, qw, qz, s, K, N, g, mi, ni)
    assert np.array_equal(ys, y64[mi, ni])      # same terms, same order


def test_per_channel_group_equals_K():
    """group_size = -1 degenerates to one group over all of K."""
    K, N = 256, 32
    qw, qz, s = _layer(K, N, K, seed=11)
    W = oracle.dequant_f64(qw, qz, s, K, N, K)
    q = oracle.awq_unpack(qw, N).astype(np.float64)
    z = oracle.awq_unpack(qz, N).astype(np.float64)
    assert np.array_equal(W, (q - z[0]) * s.view(np.float16).astype(np.float64)[0])


# ----------------------------------------------------------------------------- AWQ -> standard

def test_awq_to_standard_same_weights():
    K, N, g = 256, 96, 64
    qw, qz, s = _layer(K, N, g, seed=12)
    qw_std, qz_std = oracle.awq_to_standard(qw, qz, K, N, g)
    assert qw_std.shape == (K // 8, N)
    W_awq = oracle.dequant_f64(qw, qz, s, K, N, g)
    W_std = oracle.dequant_standard_f64(qw_std, qz_std, s, K, N, g)
    assert np.array_equal(W_awq, W_std)


def test_standard_format_closed_forms():
    """Standard order is plain: q[k, n] = k mod 8 and z[G, n] = n mod 8 give 0x76543210."""
    K, N, g = 64, 32, 32
    q = np.tile((np.arange(K) % 8)[:, None], (1, N)).astype(np.uint8)
    z = np.tile(np.arange(N) % 8, (K // g, 1)).astype(np.uint8)
    qw_std, qz_std = oracle.awq_to_standard(oracle.awq_pack(q), oracle.awq_pack(z), K, N, g)
    assert np.all(qw_std.view(np.uint32) == 0x76543210)
    assert np.all(qz_std.view(np.uint32) == 0x76543210)


# ----------------------------------------------------------------------------- [N/64][K][32 B]

def _golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                parts = line.split()
                rows[parts[0]] = parts[1:]
    return rows


def test_int4pack_layout_index_pattern():
    """code = n mod 16: byte d of every 32-byte run is (d mod 16) * 0x11 (d and d+32 agree)."""
    spec = _golden("int4pack_layout.txt")
    assert spec["block_channels"] == ["64"] and spec["run_bytes"] == ["32"]
    K, N = 8, 128
    q = np.tile(np.arange(N) % 16, (K, 1)).astype(np.uint8)
    P = oracle.int4pack_cpu(q)
    assert P.shape == (N // 64, K, 32)
    d = np.arange(32)
    assert np.all(P == ((d % 16) * 0x11).astype(np.uint8))


def test_int4pack_layout_general_pattern():
    """A pattern that separates n-block, k, d and nibble: read each nibble back by the rule."""
    K, N = 5, 192
    n = np.arange(N)
    k = np.arange(K)[:, None]
    q = ((n // 64) * 7 + k * 3 + (n % 64) // 32 * 5 + n % 32) % 16
    q = q.astype(np.uint8)
    P = oracle.int4pack_cpu(q)
    for b in range(N // 64):
        for kk in range(K):
            for dd in range(32):
                byte = int(P[b, kk, dd])
                assert byte & 0xF == q[kk, 64 * b + dd]
                assert byte >> 4 == q[kk, 64 * b + dd + 32]
    assert np.array_equal(oracle.int4unpack_cpu(P, K, N), q)


def test_int4pack_tail_N80():
    """N = 80 packs as one full 64-channel block plus a 16-channel tail (padded with 0)."""
    spec = _golden("int4pack_layout.txt")
    N, full, tail = (int(v) for v in spec["tail_N"])
    K = 16
    rng = np.random.default_rng(13)
    q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    P = oracle.int4pack_cpu(q)
    assert P.shape[0] * 64 - N == 64 - tail and N - full == tail
    assert np.array_equal(oracle.int4unpack_cpu(P, K, N), q)
    assert np.all(P[1, :, tail:] & 0xF == 0) and np.all(P[1] >> 4 == 0)


def _chunked_pack(q, chunk):
    K, N = q.shape
    out = np.zeros(((N + 63) // 64, K, 32), np.uint8)
    for n0 in range(0, N, chunk):
        oracle.int4pack_cpu(q, n0, min(n0 + chunk, N), out=out)
    return out


@pytest.mark.parametrize("shape", ["13312x2048", "2048x6656", "3072x2048", "131072x128"])
def test_int4pack_chunked_is_byte_identical(shape):
    """The page's chunk-identity shapes (N x K); the embedding is taken at K = 128 to keep the
    CPU suite short (K is the middle axis and plays no part in the chunking)."""
    spec = _golden("int4pack_layout.txt")
    N, K = (int(v) for v in shape.split("x"))
    if shape != "131072x128":
        assert shape in spec["chunk_identity_NxK"]
    rng = np.random.default_rng(N + K)
    q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    whole = oracle.int4pack_cpu(q)
    assert np.array_equal(_chunked_pack(q, 512), whole)
    ragged = 4992                                  # 78 blocks; N is not a multiple of it
    assert N % ragged != 0 or N < ragged
    assert np.array_equal(_chunked_pack(q, ragged), whole)


def test_shape_orientation_and_transients():
    """K * N * 4 bytes reproduces the page's int32 transient table, and a 512-column chunk of a
    K = 2048 matrix is the 4 MiB chunk transient: the table lists N x K."""
    t = _golden("int32_transient.txt")
    for name in ("gate_up", "down", "q_k_v", "embedding"):
        N, K, mib = (int(v) for v in t[name])
        assert K * N * 4 == mib * 2**20, name
    K, mib = int(t["chunk"][1]), int(t["chunk"][2])
    assert K * 512 * 4 == mib * 2**20
    # and the generator's shapes agree with the table
    assert inputs.SHAPES["gate_up"] == (2048, 13312)
    assert inputs.SHAPES["down"] == (6656, 2048)
    assert inputs.SHAPES["qkv"] == (2048, 3072)
    assert inputs.SHAPES["lm_head"] == (2048, 131072)


# ------------------------------------------------------------------ tied embedding gather

def _pack_awq(codes):
    """AWQ words from codes [rows][N], written out here from the slot order of the pages'
    packing (slot j of word c holds column 8c + (0, 2, 4, 6, 1, 3, 5, 7)[j])."""
    rows, N = codes.shape
    words = np.zeros((rows, N // 8), np.uint32)
    for j, col in enumerate((0, 2, 4, 6, 1, 3, 5, 7)):
        words |= codes[:, col::8].astype(np.uint32) << np.uint32(4 * j)
    return words.view(np.int32)


def test_embed_gather_closed_form():
    """Codes q[k][n] = (k + 3n) mod 16, zero 8, scale 1: every gathered value is the small
    integer ((k + 3n) mod 16) - 8, exact in fp16."""
    K, N, g = 256, 96, 64
    k = np.arange(K)[:, None]
    n = np.arange(N)[None, :]
    q = ((k + 3 * n) % 16).astype(np.uint8)
    z = np.full((K // g, N), 8, np.uint8)
    s = np.full((K // g, N), 0x3C00, np.uint16)                        # 1.0
    ids = np.array([0, 95, 7, 8, 7, 41], np.int32)                     # duplicates and both ends
    out, bad = oracle.embed_gather(_pack_awq(q), _pack_awq(z), s, K, N, g, ids)
    assert bad == 0
    want = (((np.arange(K)[None, :] + 3 * ids[:, None]) % 16) - 8).astype(np.float16)
    assert np.array_equal(out, want.view(np.uint16))


def test_embed_gather_matches_numpy_rounding():
    """Random codes, zeros and scales: each gathered value is numpy's fp16 rounding of the exact
    product (q - z) * s computed from the unpacked codes; an id outside [0, N) gives zeros."""
    K, N, g = 384, 200, 128
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = rng.integers(0, 16, (K // g, N)).astype(np.uint8)
    s = rng.uniform(1e-3, 0.05, (K // g, N)).astype(np.float16)
    ids = np.array([3, 199, -1, 120, 200, 3], np.int32)
    out, bad = oracle.embed_gather(_pack_awq(q), _pack_awq(z), s.view(np.uint16), K, N, g, ids)
    assert bad == 2
    grp = np.arange(K) // g
    for t, n in enumerate(ids):
        if 0 <= n < N:
            exact = (q[:, n].astype(np.float64) - z[grp, n]) * s[grp, n].astype(np.float64)
            assert np.array_equal(out[t], exact.astype(np.float16).view(np.uint16)), t
        else:
            assert not out[t].any()


# ------------------------------------------------------------------ bfloat16

def _bf16_widen_np(bits):
    """bfloat16 -> float64 by numpy alone: the pattern is the top half of a binary32."""
    with np.errstate(invalid="ignore"):                 # NaN patterns widen to NaN
        return (np.asarray(bits, np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


_ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)
_FIN_BF16 = _ALL_BF16[np.isfinite(_bf16_widen_np(_ALL_BF16))]
_FIN_VALS = _bf16_widen_np(_FIN_BF16)
_ORDER = np.lexsort((_FIN_BF16, _FIN_VALS))          # by value; +0 before -0 sorts by pattern


def _nearest_bf16_np(v):
    """Brute-force round-to-nearest-even into bfloat16 over the sorted finite values."""
    vals, pats = _FIN_VALS[_ORDER], _FIN_BF16[_ORDER]
    v = np.asarray(v, np.float64)
    i = np.clip(np.searchsorted(vals, v), 1, len(vals) - 1)
    lo, hi = vals[i - 1], vals[i]
    plo, phi = pats[i - 1], pats[i]
    dlo, dhi = v - lo, hi - v
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (phi % 2 == 0))
    return np.where(pick_hi, phi, plo).astype(np.uint16)


def test_bf16_widening_is_exact_for_every_pattern():
    got = oracle.bf16_bits_to_double(_ALL_BF16)
    want = _bf16_widen_np(_ALL_BF16)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_rounding_nearest_even_and_round_trip():
    # every finite pattern survives a round trip (the sign of zero included)
    assert np.array_equal(oracle.double_to_bf16_bits(_bf16_widen_np(_FIN_BF16)), _FIN_BF16)
    # midpoints between neighbours of one sign round to the even pattern
    pos = np.sort(_FIN_VALS[_FIN_VALS > 0])
    mids = (pos[:-1] + pos[1:]) / 2
    want = _nearest_bf16_np(mids)
    assert np.all(want % 2 == 0)
    assert np.array_equal(oracle.double_to_bf16_bits(mids), want)
    # random magnitudes across the whole normal and subnormal range, both signs
    rng = np.random.default_rng(11)
    v = rng.choice([-1, 1], 20000) * np.exp2(rng.uniform(-134, 127, 20000))
    assert np.array_equal(oracle.double_to_bf16_bits(v), _nearest_bf16_np(v))


def test_bf16_dequant_is_one_rounding_of_the_exact_product():
    K, N, g = 256, 64, 64
    rng = np.random.default_rng(12)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = rng.integers(0, 16, (K // g, N)).astype(np.uint8)
    sb = _nearest_bf16_np(rng.uniform(1e-3, 0.05, (K // g, N)))
    got = oracle.dequant_bf16_bits(_pack_awq(q), _pack_awq(z), sb, K, N, g)
    grp = np.arange(K) // g
    exact = (q.astype(np.float64) - z[grp]) * _bf16_widen_np(sb)[grp]
    assert np.array_equal(got, _nearest_bf16_np(exact))


def test_bf16_linear_matches_numpy_and_is_exact_on_exact_sums():
    K, N, g = 256, 48, 128
    rng = np.random.default_rng(13)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = rng.integers(0, 16, (K // g, N)).astype(np.uint8)
    sb = _nearest_bf16_np(rng.uniform(1e-3, 0.05, (K // g, N)))
    xb = _nearest_bf16_np(rng.standard_normal((3, K)))
    grp = np.arange(K) // g
    W = (q.astype(np.float64) - z[grp]) * _bf16_widen_np(sb)[grp]
    y64, yb = oracle.linear_bf16(xb, _pack_awq(q), _pack_awq(z), sb, K, N, g)
    ref = _bf16_widen_np(xb) @ W
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(yb, _nearest_bf16_np(y64))
    # x in {-2..2}, scales 2^-8: every partial sum is exact, so y is the integer product
    xi = rng.integers(-2, 3, (2, K)).astype(np.float64)
    s8 = np.full((K // g, N), 0x3B80, np.uint16)                        # bf16 2^-8
    y64, _ = oracle.linear_bf16(_nearest_bf16_np(xi), _pack_awq(q), _pack_awq(z), s8, K, N, g)
    assert np.array_equal(y64, (xi @ (q.astype(np.float64) - z[grp])) / 256.0)
