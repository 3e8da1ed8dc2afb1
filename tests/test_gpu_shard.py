"""Column-parallel split on one GPU: every rank's share, computed in turn, against the whole layer.

Each slice is repacked straight from the full AWQ tensors (their row strides) and must be byte for
byte the packed form of that slice as a layer of its own; its y must match the oracle's columns of
the whole layer (bit for bit where every partial sum is exact, else within the GEMM tolerance).
"""
import numpy as np
import pytest

from gpu_util import Layer, assert_close, awq_column_slice, dev, torch
import w4a16_group_wise_gb300 as w4
from w4a16_group_wise_gb300 import inputs, shard

pytestmark = pytest.mark.gpu


def _parts(L, world):
    return [shard.ColumnParallelLinear(L.d_qweight, L.d_qzeros, L.d_scales, L.K, L.N, L.g, r, world)
            for r in range(world)]


@pytest.mark.parametrize("name,world", [("gate_up", 2), ("gate_up", 3), ("qkv", 8), ("tail80", 2),
                                        ("down", 4)])
def test_slice_packed_bytes_equal_the_slice_as_a_layer(name, world):
    K, N = inputs.SHAPES[name]
    L = Layer(K, N, 128, seed=21)
    for p in _parts(L, world):
        if not p.width:
            continue
        qw, qz, sc = awq_column_slice(L, p.n0, p.n1)
        d = dev()
        alone = w4.repack(torch.from_numpy(qw).to(d), torch.from_numpy(qz).to(d),
                          torch.from_numpy(sc.view(np.float16)).to(d), K, p.width, L.g)
        assert torch.equal(p.packed, alone), (p.n0, p.n1)


@pytest.mark.parametrize("name,world,M", [("gate_up", 2, 1), ("gate_up", 3, 16), ("gate_up", 2, 512),
                                          ("qkv", 8, 1), ("qkv", 4, 300), ("tail80", 2, 3), ("down", 4, 64)])
def test_slices_concatenate_to_the_whole_layer(name, world, M):
    K, N = inputs.SHAPES[name]
    L = Layer(K, N, 128, seed=22)
    x_np = inputs.make_x(M, K, seed=M)
    x = torch.from_numpy(np.ascontiguousarray(x_np).view(np.uint16).view(np.int16)).to(dev()).view(torch.float16)
    ys = [p.forward(x) for p in _parts(L, world)]
    assert [y.shape[1] for y in ys] == [n1 - n0 for n0, n1 in shard.column_slices(N, world)]
    y = torch.cat(ys, dim=1)
    _, y16 = L.ref(x_np)
    assert_close(y, y16)
    if M <= 8:
        # the decode kernels add a column's chunks in an order fixed by K and the warp count, which
        # these narrower layers share with the whole one: the slices agree with it bit for bit
        whole = w4.gemm(x, L.packed, M, N, K, L.g)
        assert torch.equal(y.view(torch.int16), whole.view(torch.int16))


@pytest.mark.parametrize("M", [1, 17, 130])
def test_slices_bit_exact_when_sums_are_exact(M):
    """x in {-2..2} and s = 2^-8: every partial sum is exact, so each slice equals the oracle's
    columns bit for bit, whatever plan the narrower layer gets."""
    K, N, g = 2048, 328, 64
    L = Layer(K, N, g, seed=23)
    L.scales_bits = np.full_like(L.scales_bits, 0x1C00)          # 2^-8
    L.d_scales = torch.from_numpy(L.scales_bits.view(np.float16)).to(dev())
    xi = np.random.default_rng(M).integers(-2, 3, size=(M, K)).astype(np.float16)
    _, y16 = L.ref(xi)
    x = torch.from_numpy(xi).to(dev())
    y = torch.cat([p.forward(x) for p in _parts(L, 3)], dim=1).cpu().numpy().view(np.uint16)
    assert np.array_equal(y, y16)


@pytest.mark.parametrize("M", [1, 40])
def test_bf16_slices_concatenate_to_the_whole_layer(M):
    """The split of a bf16 layer: each rank's slice is repacked from the full bf16 scales and its
    y meets the bf16 tolerance against the oracle's columns."""
    from gpu_util import assert_close_bf16
    K, N = inputs.SHAPES["qkv"]
    L = Layer(K, N, 128, seed=24, dtype="bf16")
    x_np = inputs.make_x(M, K, seed=M, dtype="bf16")
    x = torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).to(dev()).view(torch.bfloat16)
    ys = [p.forward(x) for p in _parts(L, 3)]
    assert all(y.dtype == torch.bfloat16 for y in ys)
    y64, _ = L.ref(x_np)
    assert_close_bf16(torch.cat(ys, dim=1), y64)
    assert w4.last_device_error() == 0
