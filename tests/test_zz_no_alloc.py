"""w4a16_gemm_noalloc through the C ABI, against the oracle and against w4a16_gemm.

w4a16_gemm_noalloc serves callers that cannot allocate device memory (a runtime that plans every
buffer ahead, a host that forbids allocation after start-up, a latency-critical path): where the
tensor-core path adds split-K partial tiles through memory, it keeps them in an array built into
the library instead of a caller workspace.  That array is shared by every call and keeps the
previous call's contents, so the results are checked on two calls in a row, each element against
the CPU oracle within the tolerance of the other GEMM tests, and against the ordinary entry point.
This file is collected last on purpose.
"""
import ctypes

import pytest

from gpu_util import MAX_TOL, MEAN_TOL, Layer, assert_close, dev, errors, torch
import w4a16_group_wise_gb300 as w4
from w4a16_group_wise_gb300 import binding, inputs

P = ctypes.c_void_p


def _call(x, packed, M, N, K, g, y):
    st = P(torch.cuda.current_stream().cuda_stream)
    return binding.lib().w4a16_gemm_noalloc(P(x.data_ptr()), P(packed.data_ptr()), M, N, K, g, P(y.data_ptr()), st)


# split-K shapes (scratch in use), shapes that need none, the decode path, the N = 80 tail
CASES = [("down", 512, 128), ("qkv", 129, 128), ("qkv", 256, 128), ("qkv", 512, 128), ("square", 40, 128),
         ("gate_up", 512, 128), ("gate_up", 1, 128), ("tail80", 17, 32), ("qkv", 1, 128), ("qkv", 8, 128),
         ("lm_head", 8, 128), ("down", 24, 128), ("gate_up", 32, 64)]
# the cases that split K: under the workspace reduction they run through the built-in scratch
SPLIT = {("down", 512), ("qkv", 129), ("qkv", 256), ("square", 40)}

_refs = {}


def _layer_and_ref(name, M, g):
    """The seeded layer, x, and the oracle's fp16 y of a case (computed once per case)."""
    if (name, M, g) not in _refs:
        K, N = inputs.SHAPES[name]
        L = Layer(K, N, g, seed=21)
        x = inputs.make_x(M, K, seed=21)
        _refs[(name, M, g)] = (L, x, L.ref(x)[1])
    return _refs[(name, M, g)]


@pytest.mark.gpu
@pytest.mark.parametrize("reduction", [binding.SPLITK_AUTO, binding.SPLITK_GLOBAL])
@pytest.mark.parametrize("name,M,g", CASES)
def test_noalloc_matches_workspace_entry_point(name, M, g, reduction):
    """Under the workspace reduction the split-K shapes use the built-in scratch; under the
    default cluster reduction they need none."""
    w4.set_option(binding.OPT_SPLITK_REDUCTION, reduction)
    try:
        K, N = inputs.SHAPES[name]
        L, x_np, y16 = _layer_and_ref(name, M, g)
        x = torch.from_numpy(x_np).to(dev())
        need = w4.workspace_bytes(M, N, K, g)
        assert need <= 24 << 20  # within the built-in scratch
        if reduction == binding.SPLITK_GLOBAL and (name, M) in SPLIT:
            assert need > 0  # the case does go through the scratch
        ws_ref = w4.gemm(x, L.packed, M, N, K, g).float().cpu().numpy()
        for _ in range(2):
            y = torch.full((M, N), 3.0, dtype=torch.float16, device=dev())
            assert _call(x, L.packed, M, N, K, g, y) == binding.OK
            assert w4.last_device_error() == binding.OK
            assert_close(y, y16)  # every element against the oracle
            mx, mean = errors(y.float().cpu().numpy(), ws_ref)
            assert mx <= MAX_TOL and mean <= MEAN_TOL, (mx, mean)
    finally:
        w4.set_option(binding.OPT_SPLITK_REDUCTION, binding.SPLITK_AUTO)


def test_noalloc_rejects_bad_arguments_on_the_host():
    import __graft_entry__
    __graft_entry__.build()
    L = binding.lib()
    a, odd, nul = P(0x10000), P(0x10008), P(0)
    assert L.w4a16_gemm_noalloc(a, a, 1, 2048, 2048, 100, a, nul) == binding.ERR_UNSUPPORTED
    assert L.w4a16_gemm_noalloc(a, a, -1, 2048, 2048, 128, a, nul) == binding.ERR_INVALID
    assert L.w4a16_gemm_noalloc(nul, a, 1, 2048, 2048, 128, a, nul) == binding.ERR_INVALID
    assert L.w4a16_gemm_noalloc(odd, a, 1, 2048, 2048, 128, a, nul) == binding.ERR_MISALIGNED
    assert L.w4a16_gemm_noalloc(a, a, 0, 2048, 2048, 128, nul, nul) == binding.OK
