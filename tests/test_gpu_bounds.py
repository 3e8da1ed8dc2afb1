"""The bounds-checked debug build (_libw4a16_bounds.so: every kernel checks each global access
against its buffer's extent, records a miss in the device error word and skips the access) run
over the cases whose index arithmetic has edges: ragged M, the N = 80 tail n-block, K not a
multiple of 128, one group over all of K, the streaming wide-N decode, the split-K reductions
(cluster and workspace), the persistent tensor-core path, chunked repack, dequant, the embedding
gather and the AWQ conversion.  Every call must leave the error word clean and give the oracle's
result; the check itself is shown to fire by its self-test."""
import numpy as np
import pytest

from gpu_util import Layer, assert_close, dev, errors, torch
import oracle
import w4a16_group_wise_gb300 as w4
from w4a16_group_wise_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture
def checked():
    dev()
    with w4.bounds_checked_library():
        assert w4.bounds_checked()
        w4.last_device_error()                 # start from a clean record
        yield
        assert w4.last_device_error() == 0


def test_check_fires_in_the_debug_build_only():
    dev()
    assert not w4.bounds_checked()
    assert w4.selftest_bounds() == 0           # compiled out: nothing is judged outside
    assert w4.last_device_error() == 0
    with w4.bounds_checked_library():
        w4.last_device_error()
        assert w4.selftest_bounds() == 0x1C    # past the end, before the start, empty buffer
        assert w4.last_device_error() == w4.binding.ERR_DEVICE
        assert w4.last_device_error() == 0     # cleared, and the context is usable
        assert w4.selftest_bounds() == 0x1C


@pytest.mark.parametrize("K,N,g,Ms", [
    (6656, 80, 32, (1, 3, 12, 17, 40, 129)),   # N tail; decode at 1..16 rows, 17..32 rows, split-K, tensor core
    (224, 200, 32, (5, 20, 33)),               # K % 128 != 0, N % 64 != 0
    (96, 8, 32, (2,)),                         # a single, partly filled chunk
    (4096, 264, 64, (16, 300)),                # long K decode; ragged tensor-core tiles
    (2048, 13312, 128, (1, 8, 300)),           # gate_up: lean decode, persistent tensor core
    (6656, 2048, 128, (1, 24, 512)),           # down: 16-warp decode, 24 rows over a cluster, split-K cluster
])
def test_gemm_clean_under_bounds_checks(checked, K, N, g, Ms):
    L = Layer(K, N, g, seed=K + N)
    for M in Ms:
        x = inputs.make_x(M, K, seed=M)
        _, y16 = L.ref(x)
        assert_close(L.gemm(x), y16)
        assert w4.last_device_error() == 0, M


def test_streaming_wide_decode_clean_under_bounds_checks(checked):
    K, N = inputs.SHAPES["lm_head"]
    L = Layer(K, N, 128, seed=31)
    for M in (1, 4):
        x = inputs.make_x(M, K, seed=M)
        y = L.gemm(x).float().cpu().numpy()
        rng = np.random.default_rng(M)
        mi = rng.integers(0, M, 2048)
        ni = np.concatenate([rng.integers(0, N, 2016), np.arange(N - 32, N)])
        ref = oracle.linear_sampled(x.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, 128, mi, ni)
        ref16 = oracle.double_to_half_bits(ref).view(np.float16).astype(np.float64)
        mx, mean = errors(y[mi, ni], ref16)
        assert mx <= 2e-2 and mean <= 5e-3, (mx, mean)
        assert w4.last_device_error() == 0


def test_split_k_workspace_reduction_clean_under_bounds_checks(checked):
    K, N = inputs.SHAPES["down"]
    L = Layer(K, N, 128, seed=32)
    w4.set_option(w4.binding.OPT_SPLITK_REDUCTION, w4.binding.SPLITK_GLOBAL)
    try:
        for M in (40, 512):
            assert w4.workspace_bytes(M, N, K, 128) > 0
            x = inputs.make_x(M, K, seed=M)
            _, y16 = L.ref(x)
            assert_close(L.gemm(x), y16)
            assert w4.last_device_error() == 0
    finally:
        w4.set_option(w4.binding.OPT_SPLITK_REDUCTION, w4.binding.SPLITK_AUTO)


@pytest.mark.parametrize("K,N,gpass", [(160, 80, -1), (2048, 3072, "K")])
def test_per_channel_clean_under_bounds_checks(checked, K, N, gpass):
    g = K if gpass == "K" else -1
    L = Layer(K, N, K, seed=K)
    packed = w4.repack(L.d_qweight, L.d_qzeros, L.d_scales, K, N, g)
    W = w4.dequant(packed, K, N, g).cpu().numpy().view(np.uint16)
    assert np.array_equal(W, oracle.dequant_f16_bits(L.qweight, L.qzeros, L.scales_bits, K, N, K))
    for M in (1, 40):
        x = inputs.make_x(M, K, seed=M)
        _, y16 = oracle.linear(x.view(np.uint16), L.qweight, L.qzeros, L.scales_bits, K, N, K)
        assert_close(w4.gemm(torch.from_numpy(x).to(dev()), packed, M, N, K, g), y16)
    assert w4.last_device_error() == 0


@pytest.mark.parametrize("K,N,g", [(6656, 80, 32), (224, 200, 32), (2048, 3072, 128)])
def test_repack_dequant_embed_convert_clean_under_bounds_checks(checked, K, N, g):
    L = Layer(K, N, g, seed=K + 7)
    # chunked repack from strided column slices, 64 columns at a time
    out = torch.full_like(L.packed, 0xAB)
    for n0 in range(0, N, 64):
        n1 = min(n0 + 64, N)
        w4.repack_chunk(L.d_qweight[:, n0 // 8:n1 // 8], L.d_qzeros[:, n0 // 8:n1 // 8], L.d_scales[:, n0:n1],
                        K, N, g, n0, n1, out)
    assert torch.equal(out, L.packed)
    W = w4.dequant(L.packed, K, N, g).cpu().numpy().view(np.uint16)
    assert np.array_equal(W, oracle.dequant_f16_bits(L.qweight, L.qzeros, L.scales_bits, K, N, g))
    ids = np.array([0, N - 1, N // 2, 7, N - 1], np.int32)
    e = w4.embed(torch.from_numpy(ids).to(dev()), L.packed, K, N, g).cpu().numpy().view(np.uint16)
    ref, bad = oracle.embed_gather(L.qweight, L.qzeros, L.scales_bits, K, N, g, ids)
    assert bad == 0 and np.array_equal(e, ref)
    qs, zs = w4.awq_to_standard(L.d_qweight, L.d_qzeros, K, N, g)
    rqs, rzs = oracle.awq_to_standard(L.qweight, L.qzeros, K, N, g)
    assert np.array_equal(qs.cpu().numpy(), rqs) and np.array_equal(zs.cpu().numpy(), rzs)
    assert w4.last_device_error() == 0
