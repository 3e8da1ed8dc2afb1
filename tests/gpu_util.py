"""Helpers shared by the GPU tests: device copies of seeded layers and the tolerance check."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import w4a16_group_wise_gb300 as w4  # noqa: E402
from w4a16_group_wise_gb300 import inputs  # noqa: E402

# GEMM tolerance: max|y - y_ref| <= 2e-2 * rms(y_ref), and mean relative error
# sum|y - y_ref| / sum|y_ref| <= 5e-3, y_ref = the fp64 oracle rounded to fp16.
MAX_TOL = 2e-2
MEAN_TOL = 5e-3


def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch.device("cuda:0")


def bits_to_device(bits, dtype):
    """uint16 bit patterns (numpy) -> a CUDA tensor of the 16-bit float type `dtype`."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(dtype)


def device_bits(t):
    """A CUDA tensor of a 16-bit float type -> its bit patterns as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class Layer:
    """AWQ tensors of one layer, on the host (numpy) and on the device, plus its packed form.
    dtype "f16" (default) or "bf16": the element type of the scales, x and y."""

    def __init__(self, K, N, g, seed=0, dtype="f16", **kw):
        self.K, self.N, self.g, self.dtype = K, N, g, dtype
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float16
        h = inputs.make_weights(K, N, g, seed=seed, dtype=dtype, **kw)
        self.qweight, self.qzeros = h["qweight"], h["qzeros"]
        self.scales_bits = h["scales"].view(np.uint16)
        d = dev()
        self.d_qweight = torch.from_numpy(self.qweight).to(d)
        self.d_qzeros = torch.from_numpy(self.qzeros).to(d)
        self.d_scales = bits_to_device(self.scales_bits, self.tdtype)
        self.packed = w4.repack(self.d_qweight, self.d_qzeros, self.d_scales, K, N, g)

    def gemm(self, x_np, **kw):
        x = bits_to_device(np.ascontiguousarray(x_np).view(np.uint16), self.tdtype)
        return w4.gemm(x, self.packed, x.shape[0], self.N, self.K, self.g, **kw)

    def ref(self, x_np):
        """(y64, y bits rounded to the layer's type) from the oracle."""
        f = oracle.linear_bf16 if self.dtype == "bf16" else oracle.linear
        return f(np.ascontiguousarray(x_np).view(np.uint16), self.qweight, self.qzeros, self.scales_bits,
                 self.K, self.N, self.g)


def errors(y_gpu_f16, y_ref_f64):
    y = np.asarray(y_gpu_f16, dtype=np.float64)
    r = np.asarray(y_ref_f64, dtype=np.float64)
    d = np.abs(y - r)
    rms = np.sqrt(np.mean(r ** 2))
    return d.max() / rms, d.sum() / np.abs(r).sum()


def assert_close(y_gpu, y16_ref_bits):
    """Tolerance check of a GPU result (torch fp16) against the oracle's fp16-rounded y."""
    y = y_gpu.float().cpu().numpy()
    r = y16_ref_bits.view(np.float16).astype(np.float64)
    assert np.all(np.isfinite(y))
    mx, mean = errors(y, r)
    assert mx <= MAX_TOL, "max error %.3g rms" % mx
    assert mean <= MEAN_TOL, "mean relative error %.3g" % mean
    return mx, mean


def awq_column_slice(layer, n0, n1):
    """AWQ tensors of columns [n0, n1) (n0, n1 multiples of 8): a valid layer of its own."""
    c0, c1 = n0 // 8, n1 // 8
    return (np.ascontiguousarray(layer.qweight[:, c0:c1]), np.ascontiguousarray(layer.qzeros[:, c0:c1]),
            np.ascontiguousarray(layer.scales_bits[:, n0:n1]))


# bf16 layer tolerance, derived from its arithmetic.  Against y64 (the oracle's exact value of the
# bf16 layer, weights bf16((q - z) * s)), every output y obeys
#     |y - y64| <= 2^-8 |y64| + BF16_ABS_TOL * rms(y64)
# The first term is the final rounding to bf16 (half an ulp is at most 2^-8 of the value).  The
# second is what the kernel's fp32 value may differ by: fp32 accumulation (far below it), and on
# paths that apply a 128-row group's scale once to the exact sum of (q - z) * x, the bf16
# rounding of each weight that the oracle does and the kernel skips -- independent relative
# errors of rms about 1.6e-3, so a sum whose rms is 1.6e-3 * rms(y64); 1.5e-2 is over 9 of
# those.  The mean relative error sum|y - y64| / sum|y64| is held to 5e-3 as for fp16.
BF16_ABS_TOL = 1.5e-2


def assert_close_bf16(y_gpu, y64_ref):
    """Tolerance check of a GPU result (torch bf16) against the oracle's unrounded bf16-layer y."""
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    r = np.asarray(y64_ref, dtype=np.float64)
    assert np.all(np.isfinite(y))
    rms = np.sqrt(np.mean(r ** 2))
    d = np.abs(y - r)
    excess = d - (2.0 ** -8) * np.abs(r)
    worst = excess.max() / rms
    mean = d.sum() / np.abs(r).sum()
    assert worst <= BF16_ABS_TOL, "max error beyond the rounding term %.3g rms" % worst
    assert mean <= MEAN_TOL, "mean relative error %.3g" % mean
    return worst, mean
