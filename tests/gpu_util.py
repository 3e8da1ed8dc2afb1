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


class Layer:
    """AWQ tensors of one layer, on the host (numpy) and on the device, plus its packed form."""

    def __init__(self, K, N, g, seed=0, **kw):
        self.K, self.N, self.g = K, N, g
        h = inputs.make_weights(K, N, g, seed=seed, **kw)
        self.qweight, self.qzeros = h["qweight"], h["qzeros"]
        self.scales_bits = h["scales"].view(np.uint16)
        d = dev()
        self.d_qweight = torch.from_numpy(self.qweight).to(d)
        self.d_qzeros = torch.from_numpy(self.qzeros).to(d)
        self.d_scales = torch.from_numpy(h["scales"]).to(d)
        self.packed = w4.repack(self.d_qweight, self.d_qzeros, self.d_scales, K, N, g)

    def gemm(self, x_np, **kw):
        x = torch.from_numpy(np.ascontiguousarray(x_np)).to(self.d_qweight.device)
        return w4.gemm(x, self.packed, x.shape[0], self.N, self.K, self.g, **kw)

    def ref(self, x_np):
        """(y64, y16 bits) from the oracle."""
        return oracle.linear(x_np.view(np.uint16), self.qweight, self.qzeros, self.scales_bits,
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
