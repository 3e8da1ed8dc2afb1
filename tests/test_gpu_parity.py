"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Bars: repack and dequant bit-exact; GEMM within max|y - y_ref| <= 2e-2 * rms(y_ref) and mean
relative error <= 5e-3 (y_ref = fp64 oracle rounded to fp16), bit-exact where every partial sum
is exact, run-to-run bit-identical, and no write outside the output.
"""
import numpy as np
import pytest

from gpu_util import Layer, assert_close, awq_column_slice, dev, errors, torch
import oracle
import w4a16_group_wise_gb300 as w4
from w4a16_group_wise_gb300 import inputs

pytestmark = pytest.mark.gpu

SHAPES = inputs.SHAPES
SLOT_K = [0, 2, 4, 6, 1, 3, 5, 7]


# ------------------------------------------------------------------ dequant: bit-exact

@pytest.mark.parametrize("K,N,g", [
    (256, 128, 128), (96, 80, 32), (192, 8, 64), (384, 136, 32),
    (6656, 80, 32), (6656, 80, 64), (6656, 80, 128),
    (2048, 2048, 128), (2048, 3072, 128), (2048, 13312, 128), (6656, 2048, 128),
])
def test_dequant_bit_exact(K, N, g):
    L = Layer(K, N, g, seed=K + N + g)
    W = w4.dequant(L.packed, K, N, g)
    ref = oracle.dequant_f16_bits(L.qweight, L.qzeros, L.scales_bits, K, N, g)
    assert np.array_equal(W.cpu().numpy().view(np.uint16), ref)


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("zeros", ["sym8", "uniform"])
def test_dequant_bit_exact_edge_distributions(g, zeros):
    K, N = 6656, 80
    L = Layer(K, N, g, seed=5, zeros=zeros, scale_dist="loguniform", scale_lo=1e-4, scale_hi=0.1)
    W = w4.dequant(L.packed, K, N, g)
    ref = oracle.dequant_f16_bits(L.qweight, L.qzeros, L.scales_bits, K, N, g)
    assert np.array_equal(W.cpu().numpy().view(np.uint16), ref)


def test_dequant_lm_head_sampled_columns():
    K, N = SHAPES["lm_head"]
    L = Layer(K, N, 128, seed=3)
    W = w4.dequant(L.packed, K, N, 128)
    for n0 in (0, 65536, N - 512):
        qw, qz, s = awq_column_slice(L, n0, n0 + 512)
        ref = oracle.dequant_f16_bits(qw, qz, s, K, 512, 128)
        assert np.array_equal(W[:, n0:n0 + 512].cpu().numpy().view(np.uint16), ref)


def test_dequant_guard_bands():
    K, N, g = 384, 80, 64
    L = Layer(K, N, g, seed=1)
    buf = torch.full((K * N + 4096,), -7.0, dtype=torch.float16, device=dev())
    out = buf[2048:2048 + K * N].view(K, N)
    w4.dequant(L.packed, K, N, g, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:2048] == -7.0) and torch.all(buf[2048 + K * N:] == -7.0)


# ------------------------------------------------------------------ repack: the bytes themselves

def _decode_packed(buf, K, N, g):
    """Read the packed layout version 1 back by its written specification (include/w4a16.h)."""
    hdr = buf[:20].view(np.uint32)
    NB, KT = -(-N // 64), -(-K // 128)
    gpc = 128 // g
    CB = 4096 + gpc * 160
    body = buf[256:256 + NB * KT * CB].reshape(NB, KT, CB)
    words = np.ascontiguousarray(body[:, :, :4096]).view(np.uint32).reshape(NB, KT, 64, 16)
    q = np.zeros((KT * 128, NB * 64), np.uint8)
    for j in range(8):
        nib = ((words >> (4 * j)) & 0xF).astype(np.uint8)          # [b, t, r, w]
        for t in range(KT):
            for w in range(16):
                q[128 * t + 8 * w + SLOT_K[j], :] = nib[:, t, :, w].reshape(-1)
    meta = np.ascontiguousarray(body[:, :, 4096:]).reshape(NB, KT, gpc, 160)
    sc = np.ascontiguousarray(meta[..., :128]).view(np.uint16)     # [b, t, l, p]
    zw = np.ascontiguousarray(meta[..., 128:]).view(np.uint32)     # [b, t, l, word]
    s = np.zeros((KT * gpc, NB * 64), np.uint16)
    z = np.zeros((KT * gpc, NB * 64), np.uint8)
    for p in range(64):
        r = 16 * ((p % 8) // 2) + 8 * (p % 2) + p // 8
        for t in range(KT):
            for l in range(gpc):
                s[t * gpc + l, r::64] = sc[:, t, l, p]
                z[t * gpc + l, r::64] = (zw[:, t, l, p // 8] >> (4 * (p % 8))) & 0xF
    return hdr, q, s, z


@pytest.mark.parametrize("K,N,g", [(384, 80, 64), (256, 136, 128), (96, 72, 32)])
def test_repack_bytes_follow_documented_layout(K, N, g):
    L = Layer(K, N, g, seed=2)
    buf = L.packed.cpu().numpy()
    assert buf.size == w4.packed_bytes(K, N, g)
    hdr, q, s, z = _decode_packed(buf, K, N, g)
    assert hdr.tolist() == [0x36314134, 1, K, N, g]
    assert np.all(buf[20:256] == 0)
    assert np.array_equal(q[:K, :N], oracle.awq_unpack(L.qweight, N))
    assert np.all(q[K:] == 0) and np.all(q[:, N:] == 0)
    G = K // g
    assert np.array_equal(s[:G, :N], L.scales_bits)
    assert np.array_equal(z[:G, :N], oracle.awq_unpack(L.qzeros, N))
    assert np.all(s[G:] == 0) and np.all(s[:, N:] == 0) and np.all(z[G:] == 0) and np.all(z[:, N:] == 0)


# ------------------------------------------------------------------ chunked repack: byte-identical

def _repack_chunked(L, chunk, compact):
    K, N, g = L.K, L.N, L.g
    out = torch.full_like(L.packed, 0xAB)
    for n0 in range(0, N, chunk):
        n1 = min(n0 + chunk, N)
        qw, qz, sc = L.d_qweight[:, n0 // 8:n1 // 8], L.d_qzeros[:, n0 // 8:n1 // 8], L.d_scales[:, n0:n1]
        if compact:
            qw, qz, sc = qw.contiguous(), qz.contiguous(), sc.contiguous()
        w4.repack_chunk(qw, qz, sc, K, N, g, n0, n1, out)
    return out


@pytest.mark.parametrize("N,K", [(13312, 2048), (2048, 6656), (3072, 2048), (131072, 2048)])
def test_chunked_repack_is_byte_identical(N, K):
    L = Layer(K, N, 128, seed=4)
    for chunk in (512, 4992):                  # 4992 columns: ragged last chunk
        for compact in (False, True):
            assert torch.equal(_repack_chunked(L, chunk, compact), L.packed), (chunk, compact)


def test_chunked_repack_tail_block():
    L = Layer(6656, 80, 32, seed=4)
    assert torch.equal(_repack_chunked(L, 64, True), L.packed)


# ------------------------------------------------------------------ GEMM parity

GEMM_CASES = [
    ("square", 1), ("qkv", 1), ("gate_up", 1), ("down", 1),
    ("qkv", 16), ("gate_up", 16), ("down", 16),
    ("qkv", 3), ("gate_up", 8), ("down", 12),
    ("qkv", 512), ("gate_up", 512), ("down", 512),
    ("square", 17), ("square", 129),
    ("qkv", 32), ("gate_up", 33), ("down", 40),   # either side of the decode / tensor-core switch
]


@pytest.mark.parametrize("name,M", GEMM_CASES)
def test_gemm_layer_shapes(name, M):
    K, N = SHAPES[name]
    L = Layer(K, N, 128, seed=0)
    x = inputs.make_x(M, K, seed=0)
    _, y16 = L.ref(x)
    assert_close(L.gemm(x), y16)


@pytest.mark.parametrize("M", [1, 8, 512])
def test_gemm_lm_head_sampled(M):
    K, N = SHAPES["lm_head"]
    L = Layer(K, N, 128, seed=0)
    x = inputs.make_x(M, K, seed=1)
    y = L.gemm(x).float().cpu().numpy()
    rng = np.random.default_rng(M)
    mi = rng.integers(0, M, 4096)
    ni = np.concatenate([rng.integers(0, N, 4064), np.arange(N - 32, N)])
    ref = oracle.linear_sampled(x.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, 128, mi, ni)
    ref16 = oracle.double_to_half_bits(ref).view(np.float16).astype(np.float64)
    mx, mean = errors(y[mi, ni], ref16)
    assert mx <= 2e-2 and mean <= 5e-3, (mx, mean)


@pytest.mark.parametrize("K,N,M,g", [(2048, 7304, 1, 128), (2048, 19456, 5, 128), (4096, 7304, 8, 64),
                                     (11008, 512, 2, 128), (1024, 2440, 7, 32), (2048, 13312, 6, 128)])
def test_gemm_decode_shapes_between_the_layers(K, N, M, g):
    """Decode (M <= 8) at shapes between and around the decoder layers: a last row-tile with 8
    columns (N = 7304, 2440), a grid of row-tile pairs (N = 19456), a long K (86 chunks), several
    rows of x, groups of 32, 64 and 128.  Every output against the oracle, twice (the same bits
    both times)."""
    L = Layer(K, N, g, seed=K + N + M)
    x = inputs.make_x(M, K, seed=M)
    _, y16 = L.ref(x)
    a = L.gemm(x)
    assert_close(a, y16)
    b = L.gemm(x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("K,N,g", [(2048, 3072, 128), (2048, 3072, 32), (2048, 13312, 128), (4096, 2440, 64),
                                   (2048, 80, 32)])
def test_gemm_swizzled_x_ring_m8(K, N, g):
    """M = 8 takes the lean kernel's swizzled x ring (one-tile CTAs at N = 3072, 2440 and 80, two-tile
    CTAs at N = 13312), with the scale per chunk (g = 128) and per weight (g = 32, 64); M = 7 takes
    the plain ring.  Every output against the oracle."""
    L = Layer(K, N, g, seed=K + N + g)
    x = inputs.make_x(8, K, seed=g)
    _, y16 = L.ref(x)
    y8 = L.gemm(x)
    assert_close(y8, y16)
    y7 = L.gemm(np.ascontiguousarray(x[:7]))
    _, y16_7 = L.ref(np.ascontiguousarray(x[:7]))
    assert_close(y7, y16_7)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("N,K,M,g", [(131072, 2048, 1, 64), (131072, 2048, 4, 128), (30000, 2048, 2, 128),
                                     (30000, 2048, 3, 32), (30000, 320, 1, 64), (40000, 128, 2, 128),
                                     (30000, 2048, 5, 128), (30000, 2048, 7, 32), (131072, 2048, 8, 64)])
def test_gemm_streaming_decode_wide(N, K, M, g):
    """Decode of very wide layers (K <= 2048, more than 1824 row-tiles): resident CTAs walk pairs
    of row-tiles, prefetching the next pair's weights.  Sampled outputs against the oracle, the
    last columns (an odd row-tile count at N = 30000) included; at K = 320 and 128 most warps have
    no chunk, and K = 320 ends in a half-filled chunk."""
    L = Layer(K, N, g, seed=N + M)
    x = inputs.make_x(M, K, seed=M)
    y = L.gemm(x).float().cpu().numpy()
    assert w4.last_device_error() == 0
    rng = np.random.default_rng(N + g)
    mi = rng.integers(0, M, 4096)
    ni = np.concatenate([rng.integers(0, N, 4096 - 48), np.arange(N - 48, N)])
    ref = oracle.linear_sampled(x.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, g, mi, ni)
    ref16 = oracle.double_to_half_bits(ref).view(np.float16).astype(np.float64)
    mx, mean = errors(y[mi, ni], ref16)
    assert mx <= 2e-2 and mean <= 5e-3, (mx, mean)


def test_streaming_decode_header_mismatch_writes_nothing():
    K, N, g = 2048, 30000, 128
    L = Layer(K, N, g, seed=5)
    bad = L.packed.clone()
    bad[0] ^= 0xFF
    x = torch.from_numpy(inputs.make_x(1, K)).to(dev())
    y = torch.full((1, N), 7.0, dtype=torch.float16, device=dev())
    w4.gemm(x, bad, 1, N, K, g, y=y)
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    assert torch.all(y == 7.0)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("name,M,g", [("gate_up", 300, 128), ("gate_up", 1000, 64), ("lm_head", 200, 32),
                                     ("lm_head", 100, 128), ("lm_head", 150, 64), ("lm_head", 48, 32),
                                     ("gate_up", 777, 128), ("qkv", 1024, 128), ("qkv", 1023, 32)])
def test_gemm_persistent_ragged_sampled(name, M, g):
    """Persistent tensor-core CTAs walking several tiles each, with a ragged last m-tile (and,
    for the LM head, hundreds of n-tiles per launch); checked on sampled outputs, every row m of
    the last m-tile included.  At M <= 160 the CTAs alternate two accumulators tile by tile.  An
    odd M leaves the last row of a stored row pair alone; q_k_v at M = 1023/1024 takes one round
    of 256-row tiles (96 CTAs)."""
    K, N = SHAPES[name]
    L = Layer(K, N, g, seed=M)
    x = inputs.make_x(M, K, seed=M)
    y = L.gemm(x).float().cpu().numpy()
    rng = np.random.default_rng(M)
    mi = np.concatenate([rng.integers(0, M, 3000), np.arange(M - (M % 256 or 256), M)])
    ni = np.concatenate([rng.integers(0, N, len(mi) - 64), np.arange(N - 64, N)])
    ref = oracle.linear_sampled(x.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, g, mi, ni)
    ref16 = oracle.double_to_half_bits(ref).view(np.float16).astype(np.float64)
    mx, mean = errors(y[mi, ni], ref16)
    assert mx <= 2e-2 and mean <= 5e-3, (mx, mean)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 3, 12, 17, 27, 129])
@pytest.mark.parametrize("zeros", ["sym8", "uniform"])
def test_gemm_edge_tail(g, M, zeros):
    K, N = SHAPES["tail80"]
    L = Layer(K, N, g, seed=M, zeros=zeros, scale_dist="loguniform", scale_lo=1e-4, scale_hi=0.1)
    x = inputs.make_x(M, K, seed=M)
    _, y16 = L.ref(x)
    assert_close(L.gemm(x), y16)


@pytest.mark.parametrize("K,N,g,M", [(96, 8, 32, 5), (192, 72, 64, 2), (128, 64, 128, 1),
                                     (224, 200, 32, 33), (4096, 264, 64, 16), (2048, 200, 32, 13),
                                     (224, 200, 32, 9), (2048, 13312, 128, 11), (1024, 2440, 64, 16)])
def test_gemm_small_ragged(K, N, g, M):
    L = Layer(K, N, g, seed=7)
    x = inputs.make_x(M, K, seed=7)
    _, y16 = L.ref(x)
    assert_close(L.gemm(x), y16)


@pytest.mark.parametrize("M", [1, 4, 5, 8, 9, 12, 16, 17, 21, 32, 33, 130])
@pytest.mark.parametrize("g", [32, 128])
def test_gemm_bit_exact_when_sums_are_exact(M, g):
    """x in {-2..2} and s = 2^-8: every product and fp32 partial sum is exact, so the result must
    equal the oracle bit for bit, whatever the summation order."""
    K, N = 2048, 192
    L = Layer(K, N, g, seed=8)
    L.scales_bits = np.full_like(L.scales_bits, 0x1C00)          # 2^-8
    L.d_scales = torch.from_numpy(L.scales_bits.view(np.float16)).to(dev())
    L.packed = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales, K, N, g)
    xi = np.random.default_rng(M).integers(-2, 3, size=(M, K)).astype(np.float16)
    _, y16 = L.ref(xi)
    y = L.gemm(xi).cpu().numpy().view(np.uint16)
    assert np.array_equal(y, y16)


@pytest.mark.parametrize("N,K,M,g", [(30000, 2048, 1, 128), (30000, 2048, 4, 128), (30000, 2048, 8, 32),
                                     (13312, 2048, 512, 128), (13312, 2048, 777, 64)])
def test_gemm_bit_exact_when_sums_are_exact_wide(N, K, M, g):
    """The exact-sum pin above on the paths its 192-column layer does not reach: the streaming
    decode (more than 1824 row-tiles: resident CTAs walking row-tile pairs) and the persistent
    tensor-core path (gate_up at M = 512 and 777: several tiles per CTA, the last one drained by
    all warps).  x in {-2..2} and s = 2^-8 keep every product and fp32 partial sum exact, so the
    sampled outputs (the last columns included) must equal the oracle's bit for bit."""
    L = Layer(K, N, g, seed=M + N)
    L.scales_bits = np.full_like(L.scales_bits, 0x1C00)          # 2^-8
    L.d_scales = torch.from_numpy(L.scales_bits.view(np.float16)).to(dev())
    L.packed = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales, K, N, g)
    xi = np.random.default_rng(M + 1).integers(-2, 3, size=(M, K)).astype(np.float16)
    y = L.gemm(xi).cpu().numpy().view(np.uint16)
    assert w4.last_device_error() == 0
    rng = np.random.default_rng(N + M)
    mi = rng.integers(0, M, 4096)
    ni = np.concatenate([rng.integers(0, N, 4096 - 64), np.arange(N - 64, N)])
    ref = oracle.linear_sampled(xi.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, g, mi, ni)
    assert np.array_equal(y[mi, ni], oracle.double_to_half_bits(ref))


def test_gemm_q_equal_z_gives_zero():
    K, N, g = 1024, 256, 64
    L = Layer(K, N, g, seed=9)
    L.qweight = np.repeat(L.qzeros, g, axis=0)
    L.d_qweight = torch.from_numpy(L.qweight).to(dev())
    L.packed = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales, K, N, g)
    for M in (1, 16, 64):
        y = L.gemm(inputs.make_x(M, K, seed=M))
        assert torch.all(y == 0)


@pytest.mark.parametrize("name,M,g", [("qkv", 17, 128), ("gate_up", 20, 128), ("down", 24, 128),
                                     ("gate_up", 22, 64), ("qkv", 32, 32), ("down", 31, 64), ("square", 29, 128)])
def test_gemm_mid_rows_one_pass(name, M, g):
    """17..32 rows: one pass over the weights, x staged once per CTA and K split over a cluster
    of CTAs whose partials are added in rank order; down's 52 chunks leave a short last split,
    and g = 32 / 64 scale each weight before the products."""
    K, N = SHAPES[name]
    L = Layer(K, N, g, seed=M)
    x = inputs.make_x(M, K, seed=M)
    _, y16 = L.ref(x)
    assert_close(L.gemm(x), y16)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("K,N,g,M", [(160, 80, 32, 19), (224, 136, 32, 32), (6656, 80, 128, 25),
                                     (4096, 264, 64, 18), (96, 8, 32, 23)])
def test_gemm_mid_rows_ragged(K, N, g, M):
    """17..32 rows with K not a multiple of 128, N not a multiple of 64, and fewer chunks than
    splits would like."""
    L = Layer(K, N, g, seed=K + M)
    x = inputs.make_x(M, K, seed=M)
    _, y16 = L.ref(x)
    assert_close(L.gemm(x), y16)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("M", [1, 16, 24, 512])
def test_gemm_deterministic(M):
    K, N = SHAPES["gate_up"]
    L = Layer(K, N, 128, seed=10)
    x = inputs.make_x(M, K, seed=10)
    a, b = L.gemm(x), L.gemm(x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,N", [(3, 80), (17, 80), (129, 136), (1, 2048)])
def test_gemm_guard_bands(M, N):
    K, g = 512, 64
    L = Layer(K, N, g, seed=11)
    buf = torch.full((M * N + 8192,), 1234.0, dtype=torch.float16, device=dev())
    y = buf[4096:4096 + M * N].view(M, N)
    x = inputs.make_x(M, K, seed=11)
    L.gemm(x, y=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:4096] == 1234.0) and torch.all(buf[4096 + M * N:] == 1234.0)
    _, y16 = L.ref(x)
    assert_close(y, y16)


def test_gemm_m0_is_noop():
    L = Layer(256, 64, 128, seed=12)
    y = torch.full((1, 64), 5.0, dtype=torch.float16, device=dev())
    x = torch.zeros((1, 256), dtype=torch.float16, device=dev())
    w4.gemm(x, L.packed, 0, 64, 256, 128, y=y)
    torch.cuda.synchronize()
    assert torch.all(y == 5.0)


def test_header_mismatch_is_reported_and_nothing_written():
    K, N, g = 512, 128, 128
    L = Layer(K, N, g, seed=13)
    assert w4.last_device_error() == 0
    bad = L.packed.clone()
    bad[0] ^= 0xFF                                       # corrupt the magic
    # the lean decode kernel, the 16-row kernel, the one-pass mid-size kernel (a cluster of K
    # splits that all see the bad header), the tensor-core kernel
    for Mb in (1, 12, 24, 40):
        xb = torch.from_numpy(inputs.make_x(Mb, K)).to(dev())
        yb = torch.full((Mb, N), 7.0, dtype=torch.float16, device=dev())
        w4.gemm(xb, bad, Mb, N, K, g, y=yb)
        assert w4.last_device_error() == w4.binding.ERR_DEVICE, Mb
        assert torch.all(yb == 7.0), Mb
    x = torch.from_numpy(inputs.make_x(2, K)).to(dev())
    y = torch.full((2, N), 7.0, dtype=torch.float16, device=dev())
    w4.gemm(x, bad, 2, N, K, g, y=y)
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    assert torch.all(y == 7.0)
    W = torch.full((K, N), 7.0, dtype=torch.float16, device=dev())
    w4.dequant(bad, K, N, g, out=W)
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    assert torch.all(W == 7.0)
    # a smaller N than the buffer was packed for is also caught (and reads stay in bounds)
    w4.gemm(x, L.packed, 2, 64, K, g, y=y[:, :64].contiguous())
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    # the record is cleared and a correct call runs clean
    y_ok = w4.gemm(x, L.packed, 2, N, K, g)
    assert w4.last_device_error() == 0
    _, y16 = L.ref(x.cpu().numpy())
    assert_close(y_ok, y16)


def test_bounded_waits_time_out_and_the_context_stays_usable():
    """Failure detection without a fault: the library's bounded waits, on a barrier that never
    completes, give up after the limit and record the timeout; the context keeps working."""
    assert w4.last_device_error() == 0
    assert w4.binding.selftest_wait_timeout(1_000_000) == 3   # both the polling and the sleeping wait
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    assert w4.last_device_error() == 0                        # the record is cleared
    K, N, g = 512, 128, 128
    L = Layer(K, N, g, seed=40)
    for M in (3, 64):
        x = inputs.make_x(M, K, seed=M)
        _, y16 = L.ref(x)
        assert_close(L.gemm(x), y16)
    assert w4.last_device_error() == 0


def test_nondefault_stream():
    K, N, g = 2048, 3072, 128
    L = Layer(K, N, g, seed=14)
    x = inputs.make_x(4, K, seed=14)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xd = torch.from_numpy(x).to(dev())
        y = w4.gemm(xd, L.packed, 4, N, K, g)
    s.synchronize()
    _, y16 = L.ref(x)
    assert_close(y, y16)


@pytest.mark.parametrize("K,N,g,M", [(4096, 19456, 128, 1), (4096, 19456, 64, 16), (8192, 20480, 32, 3)])
def test_gemm_long_k_ring_refill(K, N, g, M):
    """Enough n-blocks that K is not split and more chunks per CTA than shared-memory ring slots,
    so ring slots are refilled; checked on sampled outputs."""
    L = Layer(K, N, g, seed=15)
    x = inputs.make_x(M, K, seed=15)
    y = L.gemm(x).float().cpu().numpy()
    rng = np.random.default_rng(15)
    mi = rng.integers(0, M, 3000)
    ni = np.concatenate([rng.integers(0, N, 2936), np.arange(64), np.arange(N - 64, N)])[:3000]
    ref = oracle.linear_sampled(x.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, g, mi, ni)
    ref16 = oracle.double_to_half_bits(ref).view(np.float16).astype(np.float64)
    mx, mean = errors(y[mi, ni], ref16)
    assert mx <= 2e-2 and mean <= 5e-3, (mx, mean)


@pytest.fixture
def splitk_global():
    """The workspace reduction of split-K partial tiles for the duration of a test."""
    w4.set_option(w4.binding.OPT_SPLITK_REDUCTION, w4.binding.SPLITK_GLOBAL)
    yield
    w4.set_option(w4.binding.OPT_SPLITK_REDUCTION, w4.binding.SPLITK_AUTO)


@pytest.mark.parametrize("name,M", [("down", 512), ("qkv", 129), ("square", 40)])
def test_gemm_split_k_workspace_reuse(name, M, splitk_global):
    """Where the tensor-core path splits K, one zero-filled workspace serves call after call:
    every completed call leaves its arrival counters at zero, and results are bit-identical."""
    K, N = SHAPES[name]
    L = Layer(K, N, 128, seed=16)
    need = w4.workspace_bytes(M, N, K, 128)
    assert need > 0, "expected a split-K plan for this shape"
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device=dev())   # partials need no init
    ws[:4096] = 0
    x = inputs.make_x(M, K, seed=16)
    ys = [L.gemm(x, workspace=ws) for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
    torch.cuda.synchronize()
    # the arrival counters (first 4096 bytes) are all back to zero
    assert int(torch.count_nonzero(ws[:4096])) == 0
    _, y16 = L.ref(x)
    assert_close(ys[0], y16)


def test_gemm_workspace_too_small_is_rejected(splitk_global):
    K, N = SHAPES["down"]
    L = Layer(K, N, 128, seed=17)
    M = 512
    need = w4.workspace_bytes(M, N, K, 128)
    assert need > 0
    small = torch.zeros(need - 16, dtype=torch.uint8, device=dev())
    x = torch.from_numpy(inputs.make_x(M, K)).to(dev())
    with pytest.raises(w4.W4A16Error) as e:
        w4.gemm(x, L.packed, M, N, K, 128, workspace=small)
    assert e.value.status == w4.binding.ERR_WORKSPACE


@pytest.mark.parametrize("name,M", [("down", 512), ("qkv", 256), ("qkv", 129), ("square", 40), ("down", 64),
                                    ("down", 40)])
def test_gemm_split_k_cluster_matches_workspace_reduction(name, M):
    """The cluster reduction (distributed shared memory, no workspace) and the workspace
    reduction add the same partial tiles in the same order: bit-identical y, close to the oracle."""
    K, N = SHAPES[name]
    L = Layer(K, N, 128, seed=18)
    x = inputs.make_x(M, K, seed=18)
    assert w4.workspace_bytes(M, N, K, 128) == 0, "a GB300 runs the split-K clusters: no workspace"
    y_cluster = L.gemm(x)
    w4.set_option(w4.binding.OPT_SPLITK_REDUCTION, w4.binding.SPLITK_GLOBAL)
    try:
        need = w4.workspace_bytes(M, N, K, 128)
        assert need > 0, "expected a split-K plan for this shape"
        ws = torch.zeros(need, dtype=torch.uint8, device=dev())
        y_global = L.gemm(x, workspace=ws)
    finally:
        w4.set_option(w4.binding.OPT_SPLITK_REDUCTION, w4.binding.SPLITK_AUTO)
    assert torch.equal(y_cluster.view(torch.int16), y_global.view(torch.int16))
    assert w4.last_device_error() == 0
    _, y16 = L.ref(x)
    assert_close(y_cluster, y16)


# ------------------------------------------------------------------ tied embedding gather

@pytest.mark.parametrize("name,g,T", [("lm_head", 128, 300), ("tail80", 32, 40), ("square", 64, 7)])
def test_embed_gather_bit_exact(name, g, T):
    """Rows of the quantized tied embedding equal the oracle's gather bit for bit: duplicate ids,
    the first and last columns, and (N = 80) columns of the 16-wide tail n-block."""
    K, N = SHAPES[name]
    L = Layer(K, N, g, seed=T)
    rng = np.random.default_rng(T)
    ids = np.concatenate([rng.integers(0, N, T - 4), [0, N - 1, N - 1, N // 2]]).astype(np.int32)
    if N % 64:
        ids[:8] = np.arange(N - 16, N - 8)                    # the tail block
    out = w4.embed(torch.from_numpy(ids).to(dev()), L.packed, K, N, g).cpu().numpy().view(np.uint16)
    ref, bad = oracle.embed_gather(L.qweight, L.qzeros, L.scales_bits, K, N, g, ids)
    assert bad == 0
    assert np.array_equal(out, ref)
    assert w4.last_device_error() == 0


def test_embed_gather_ragged_k():
    """K not a multiple of 128 (g = 32): the last chunk holds only part of its rows."""
    K, N, g = 160, 192, 32
    L = Layer(K, N, g, seed=3)
    ids = np.array([5, 191, 64, 63, 0], np.int32)
    out = w4.embed(torch.from_numpy(ids).to(dev()), L.packed, K, N, g).cpu().numpy().view(np.uint16)
    ref, _ = oracle.embed_gather(L.qweight, L.qzeros, L.scales_bits, K, N, g, ids)
    assert np.array_equal(out, ref)


def test_embed_out_of_range_id_gives_zeros_and_an_error():
    K, N = SHAPES["square"]
    L = Layer(K, N, 128, seed=4)
    ids = np.array([7, N, -3, 9], np.int32)
    out = torch.full((4, K), 1.0, dtype=torch.float16, device=dev())
    w4.embed(torch.from_numpy(ids).to(dev()), L.packed, K, N, 128, out=out)
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    o = out.cpu().numpy().view(np.uint16)
    ref, bad = oracle.embed_gather(L.qweight, L.qzeros, L.scales_bits, K, N, 128, ids)
    assert bad == 2 and np.array_equal(o, ref)
    assert w4.last_device_error() == 0                      # the record was cleared


def test_embed_header_mismatch_writes_nothing():
    K, N = SHAPES["square"]
    L = Layer(K, N, 128, seed=5)
    ids = torch.tensor([1, 2, 3], dtype=torch.int32, device=dev())
    out = torch.full((3, 1024), 7.0, dtype=torch.float16, device=dev())
    w4.embed(ids, L.packed, 1024, N, 128, out=out)          # K disagrees with the packed header
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    assert bool((out == 7.0).all())


def test_embed_empty_is_noop():
    K, N = SHAPES["square"]
    L = Layer(K, N, 128, seed=6)
    out = w4.embed(torch.empty(0, dtype=torch.int32, device=dev()), L.packed, K, N, 128)
    assert out.shape == (0, K)


# ------------------------------------------------------------------ per-channel groups

@pytest.mark.parametrize("K,N", [(2048, 3072), (192, 136), (160, 80)])
@pytest.mark.parametrize("gpass", ["K", -1])
def test_per_channel_groups(K, N, gpass):
    """One group over all of K (the pages' group_size = -1): repacked from one row of scales and
    zeros, the dequantized weights are bit-exact and the GEMM (decode and tensor-core paths)
    meets the tolerance, against the oracle run with g = K."""
    g = K if gpass == "K" else -1
    L = Layer(K, N, K, seed=K + N)                      # qzeros [1][N/8], scales [1][N]
    packed = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales, K, N, g)
    W = w4.dequant(packed, K, N, g).cpu().numpy().view(np.uint16)
    assert np.array_equal(W, oracle.dequant_f16_bits(L.qweight, L.qzeros, L.scales_bits, K, N, K))
    for M in (1, 24, 40, 300):
        x = inputs.make_x(M, K, seed=M)
        y = w4.gemm(torch.from_numpy(x).to(dev()), packed, M, N, K, g)
        _, y16 = oracle.linear(x.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, K)
        assert_close(y, y16)
    ids = np.array([0, N - 1, 3, 3], np.int32)
    e = w4.embed(torch.from_numpy(ids).to(dev()), packed, K, N, g).cpu().numpy().view(np.uint16)
    ref, _ = oracle.embed_gather(L.qweight, L.qzeros, L.scales_bits, K, N, K, ids)
    assert np.array_equal(e, ref)
    assert w4.last_device_error() == 0


# ------------------------------------------------------------------ AWQ -> standard packing

@pytest.mark.parametrize("K,N,g", [(2048, 3072, 128), (6656, 80, 32), (192, 136, 192), (160, 80, -1)])
def test_awq_to_standard_bit_exact(K, N, g):
    """The GPU conversion to the GPTQ-style standard packing equals the oracle's word for word
    (N = 80 tail, per-channel groups passed as g = K and as g = -1)."""
    L = Layer(K, N, K if g == -1 else g, seed=K + N + 1)
    qs, zs = w4.awq_to_standard(L.d_qweight, L.d_qzeros, K, N, g)
    rqs, rzs = oracle.awq_to_standard(L.qweight, L.qzeros, K, N, K if g == -1 else g)
    assert np.array_equal(qs.cpu().numpy(), rqs)
    assert np.array_equal(zs.cpu().numpy(), rzs)
