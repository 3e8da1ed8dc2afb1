"""GPU parity of the bfloat16 layer (scales, x, W and y in bf16) against the CPU oracle.

Bars: repack and dequant bit-exact; GEMM within the bf16 tolerance of gpu_util (the final
rounding plus 1.5e-2 rms), bit-exact where every partial sum is exact; a packed buffer of one
element type is refused by the calls of the other.
"""
import numpy as np
import pytest

from gpu_util import Layer, assert_close_bf16, bits_to_device, dev, device_bits, torch
import oracle
import w4a16_group_wise_gb300 as w4
from w4a16_group_wise_gb300 import inputs

pytestmark = pytest.mark.gpu

SHAPES = inputs.SHAPES


@pytest.mark.parametrize("K,N,g", [(256, 128, 128), (96, 80, 32), (384, 136, 64), (6656, 80, 32),
                                   (6656, 80, 128), (2048, 3072, 128), (6656, 2048, 64)])
def test_dequant_bf16_bit_exact(K, N, g):
    L = Layer(K, N, g, seed=K + N, dtype="bf16")
    W = w4.dequant(L.packed, K, N, g, dtype=torch.bfloat16)
    ref = oracle.dequant_bf16_bits(L.qweight, L.qzeros, L.scales_bits, K, N, g)
    assert np.array_equal(device_bits(W), ref)


@pytest.mark.parametrize("g", [32, 128])
def test_dequant_bf16_wide_scale_range(g):
    """Log-uniform scales over three decades: every bf16 exponent path of the one rounding."""
    K, N = 6656, 80
    L = Layer(K, N, g, seed=2, dtype="bf16", zeros="sym8", scale_dist="loguniform", scale_lo=1e-4,
              scale_hi=0.1)
    W = w4.dequant(L.packed, K, N, g, dtype=torch.bfloat16)
    ref = oracle.dequant_bf16_bits(L.qweight, L.qzeros, L.scales_bits, K, N, g)
    assert np.array_equal(device_bits(W), ref)


def test_bf16_packing_differs_from_fp16_only_in_the_dtype_word():
    """The scales are copied as bit patterns: a bf16 repack equals the fp16 repack of the same
    bits except for the header's dtype word (bytes 20..23)."""
    K, N, g = 384, 136, 64
    L = Layer(K, N, g, seed=3, dtype="bf16")
    p16 = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales.view(torch.float16), K, N, g)
    a, b = L.packed.cpu().numpy(), p16.cpu().numpy()
    assert a[20:24].view(np.int32)[0] == 1 and b[20:24].view(np.int32)[0] == 0
    a[20:24] = 0
    assert np.array_equal(a, b)


def test_bf16_chunked_repack_is_byte_identical():
    K, N = SHAPES["gate_up"]
    L = Layer(K, N, 128, seed=4, dtype="bf16")
    out = torch.zeros_like(L.packed)
    for n0 in range(0, N, 4096):
        n1 = min(N, n0 + 4096)
        w4.binding.repack_chunk(L.d_qweight[:, n0 // 8:n1 // 8], L.d_qzeros[:, n0 // 8:n1 // 8],
                                L.d_scales[:, n0:n1], K, N, 128, n0, n1, out)
    assert torch.equal(out, L.packed)


GEMM_CASES = [
    ("square", 1), ("qkv", 1), ("gate_up", 1), ("down", 1),
    ("qkv", 3), ("gate_up", 16), ("down", 12), ("qkv", 8), ("gate_up", 8), ("qkv", 16), ("square", 10),
    ("qkv", 32), ("gate_up", 33), ("down", 40), ("down", 24), ("gate_up", 20),
    ("qkv", 512), ("gate_up", 512), ("down", 512), ("square", 129),
]


@pytest.mark.parametrize("name,M", GEMM_CASES)
def test_gemm_bf16_layer_shapes(name, M):
    K, N = SHAPES[name]
    L = Layer(K, N, 128, seed=5, dtype="bf16")
    x = inputs.make_x(M, K, seed=5, dtype="bf16")
    y64, _ = L.ref(x)
    y = L.gemm(x)
    assert y.dtype == torch.bfloat16
    assert_close_bf16(y, y64)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 3, 17, 129])
def test_gemm_bf16_edge_tail(g, M):
    K, N = SHAPES["tail80"]
    L = Layer(K, N, g, seed=M, dtype="bf16", scale_dist="loguniform", scale_lo=1e-4, scale_hi=0.1)
    x = inputs.make_x(M, K, seed=M, dtype="bf16")
    y64, _ = L.ref(x)
    assert_close_bf16(L.gemm(x), y64)


@pytest.mark.parametrize("K,N,g,M", [(96, 8, 32, 5), (192, 72, 64, 2), (224, 200, 32, 33)])
def test_gemm_bf16_small_ragged(K, N, g, M):
    L = Layer(K, N, g, seed=7, dtype="bf16")
    x = inputs.make_x(M, K, seed=7, dtype="bf16")
    y64, _ = L.ref(x)
    assert_close_bf16(L.gemm(x), y64)


@pytest.mark.parametrize("M", [1, 4, 8, 16, 20, 32, 33, 130])
@pytest.mark.parametrize("g", [32, 128])
def test_gemm_bf16_bit_exact_when_sums_are_exact(M, g):
    """x in {-2..2} and s = 2^-8: every product and fp32 partial sum is exact, so both sides
    round the same exact value once to bf16 and must agree bit for bit."""
    K, N = 2048, 192
    L = Layer(K, N, g, seed=8, dtype="bf16")
    L.scales_bits = np.full_like(L.scales_bits, 0x3B80)          # 2^-8 in bf16
    L.d_scales = bits_to_device(L.scales_bits, torch.bfloat16)
    L.packed = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales, K, N, g)
    xi = inputs.bf16_bits(np.random.default_rng(M).integers(-2, 3, size=(M, K)))
    _, yb = L.ref(xi)
    assert np.array_equal(device_bits(L.gemm(xi)), yb)


@pytest.mark.parametrize("N,K,M,g", [(30000, 2048, 1, 128), (30000, 2048, 8, 32), (13312, 2048, 512, 128)])
def test_gemm_bf16_bit_exact_when_sums_are_exact_wide(N, K, M, g):
    """The wide exact-sum pin of the fp16 suite for a bf16 layer: the streaming decode (30000
    columns) and the persistent tensor-core path (gate_up at M = 512).  x in {-2..2} and s = 2^-8
    are exact in fp16 and bf16 alike, so the exact sums are those of the oracle's sampled product
    over the same values, rounded once to bf16; the sampled outputs must match bit for bit."""
    L = Layer(K, N, g, seed=M + N, dtype="bf16")
    L.scales_bits = np.full_like(L.scales_bits, 0x3B80)          # 2^-8 in bf16
    L.d_scales = bits_to_device(L.scales_bits, torch.bfloat16)
    L.packed = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales, K, N, g)
    xi_int = np.random.default_rng(M + 2).integers(-2, 3, size=(M, K))
    y = device_bits(L.gemm(inputs.bf16_bits(xi_int)))
    assert w4.last_device_error() == 0
    rng = np.random.default_rng(N + M + 1)
    mi = rng.integers(0, M, 4096)
    ni = np.concatenate([rng.integers(0, N, 4096 - 64), np.arange(N - 64, N)])
    s16 = np.full_like(L.scales_bits, 0x1C00)                    # the same 2^-8 in fp16
    ref = oracle.linear_sampled(xi_int.astype(np.float16).view(np.uint16), L.qweight, L.qzeros, s16, K, N, g,
                                mi, ni)
    assert np.array_equal(y[mi, ni], oracle.double_to_bf16_bits(ref))


@pytest.mark.parametrize("M", [1, 512])
def test_gemm_bf16_deterministic(M):
    K, N = SHAPES["gate_up"]
    L = Layer(K, N, 128, seed=10, dtype="bf16")
    x = inputs.make_x(M, K, seed=10, dtype="bf16")
    a, b = L.gemm(x), L.gemm(x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_element_type_mismatch_is_reported_and_nothing_written():
    K, N, g = 512, 128, 128
    Lb = Layer(K, N, g, seed=11, dtype="bf16")
    Lh = Layer(K, N, g, seed=11)
    assert w4.last_device_error() == 0
    for M in (2, 64):
        # an fp16 buffer given to the bf16 GEMM, and a bf16 buffer to the fp16 GEMM
        xb = bits_to_device(inputs.make_x(M, K, dtype="bf16"), torch.bfloat16)
        yb = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=dev())
        w4.gemm(xb, Lh.packed, M, N, K, g, y=yb)
        assert w4.last_device_error() == w4.binding.ERR_DEVICE
        assert torch.all(yb == 7.0)
        xh = torch.from_numpy(inputs.make_x(M, K)).to(dev())
        yh = torch.full((M, N), 7.0, dtype=torch.float16, device=dev())
        w4.gemm(xh, Lb.packed, M, N, K, g, y=yh)
        assert w4.last_device_error() == w4.binding.ERR_DEVICE
        assert torch.all(yh == 7.0)
    W = torch.full((K, N), 7.0, dtype=torch.float16, device=dev())
    w4.dequant(Lb.packed, K, N, g, out=W)
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    assert torch.all(W == 7.0)
    e = torch.full((3, K), 7.0, dtype=torch.bfloat16, device=dev())
    w4.embed(torch.tensor([0, 5, 9], dtype=torch.int32, device=dev()), Lh.packed, K, N, g, out=e)
    assert w4.last_device_error() == w4.binding.ERR_DEVICE
    assert torch.all(e == 7.0)


@pytest.mark.parametrize("name,g,T", [("lm_head", 128, 300), ("tail80", 32, 40)])
def test_embed_bf16_bit_exact(name, g, T):
    K, N = SHAPES[name]
    L = Layer(K, N, g, seed=12, dtype="bf16")
    ids = np.random.default_rng(T).integers(0, N, T).astype(np.int32)
    ids[:2] = (0, N - 1)
    out = w4.embed(torch.from_numpy(ids).to(dev()), L.packed, K, N, g, dtype=torch.bfloat16)
    c = np.unique(ids // 8)
    ref_w = oracle.dequant_bf16_bits(L.qweight[:, c], L.qzeros[:, c],
                                     L.scales_bits.reshape(-1, N // 8, 8)[:, c].reshape(-1, 8 * len(c)),
                                     K, 8 * len(c), g)
    pos = {cc: i for i, cc in enumerate(c)}
    ref = np.stack([ref_w[:, 8 * pos[n // 8] + n % 8] for n in ids])
    assert np.array_equal(device_bits(out), ref)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("gpass", ["K", -1])
def test_gemm_bf16_per_channel(gpass):
    """One group over all of K, in bf16: the same as the g = 128 layer whose every group carries
    the column's one scale and zero."""
    K, N = 2048, 3072
    g = K if gpass == "K" else -1
    h = inputs.make_weights(K, N, K, seed=13, dtype="bf16")
    qw, qz, s = h["qweight"], h["qzeros"], h["scales"].view(np.uint16)
    d = dev()
    packed = w4.repack(torch.from_numpy(qw).to(d), torch.from_numpy(qz).to(d), bits_to_device(s, torch.bfloat16),
                       K, N, g)
    G = K // 128
    for M in (1, 64):
        x = inputs.make_x(M, K, seed=M, dtype="bf16")
        y = w4.gemm(bits_to_device(x, torch.bfloat16), packed, M, N, K, g)
        y64, _ = oracle.linear_bf16(x, qw, np.repeat(qz, G, axis=0), np.repeat(s, G, axis=0), K, N, 128)
        assert_close_bf16(y, y64)
