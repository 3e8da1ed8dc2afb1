"""Seeded synthetic inputs for the W4A16 group-wise linear layer.

This module holds none of the layer's arithmetic: it only draws random tensors with the
shapes and value distributions of the pages' layers, and both the CUDA path (tests, bench)
and the CPU oracle (tests, cpu baseline) consume what it returns.

Recipe (numpy PCG64; one independent sub-stream per tensor from a SeedSequence keyed by
(seed, tensor tag, shape)):
  - qweight int32 [K, N/8] and qzeros int32 [K/g, N/8]: uniform random 32-bit words.  Every
    nibble of a uniform word is an independent uniform 4-bit code 0..15, so no packing order
    is involved.  ``zeros="sym8"`` gives every zero code 8 (word 0x88888888).
  - scales fp16 [K/g, N]: uniform on [lo, hi] (default [0.002, 0.02]) or log-uniform on
    [lo, hi] (``scale_dist="loguniform"``, e.g. [1e-4, 0.1]), rounded to fp16 by numpy.
  - x fp16 [M, K]: standard normal, rounded to fp16 by numpy.
  - bf16 layers (``dtype="bf16"``): the same draws, scales and x rounded to bfloat16 by torch
    (nearest even) and returned as uint16 bit patterns, numpy having no bfloat16 type.
Shapes follow the pages' layers: K = 2048 hidden, q_k_v N = 3072, gate_up N = 13312,
down K = 6656 / N = 2048, tied embedding / LM head N = 131072, and the N = 80 tail case.
"""
import numpy as np

_TAGS = {"qweight": 1, "qzeros": 2, "scales": 3, "x": 4}


def _rng(seed, tag, *shape):
    ss = np.random.SeedSequence([int(seed), _TAGS[tag]] + [int(s) for s in shape])
    return np.random.Generator(np.random.PCG64(ss))


def bf16_bits(a):
    """float array -> bfloat16 bit patterns (uint16 array of the same shape), rounded by torch."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def make_weights(K, N, g, seed=0, zeros="uniform", scale_dist="uniform", scale_lo=0.002,
                 scale_hi=0.02, dtype="f16"):
    """AWQ-format tensors of one layer: dict(qweight int32, qzeros int32, scales) with scales
    float16, or (dtype="bf16") bfloat16 bits as uint16."""
    if N % 8 or K % g:
        raise ValueError("N must be a multiple of 8 and K a multiple of g")
    G = K // g
    qweight = _rng(seed, "qweight", K, N, g).integers(0, 2**32, size=(K, N // 8),
                                                      dtype=np.uint32).view(np.int32)
    if zeros == "uniform":
        qzeros = _rng(seed, "qzeros", K, N, g).integers(0, 2**32, size=(G, N // 8),
                                                        dtype=np.uint32).view(np.int32)
    elif zeros == "sym8":
        qzeros = np.full((G, N // 8), 0x88888888, np.uint32).view(np.int32)
    else:
        raise ValueError(zeros)
    r = _rng(seed, "scales", K, N, g)
    if scale_dist == "uniform":
        s = r.uniform(scale_lo, scale_hi, size=(G, N))
    elif scale_dist == "loguniform":
        s = np.exp(r.uniform(np.log(scale_lo), np.log(scale_hi), size=(G, N)))
    else:
        raise ValueError(scale_dist)
    scales = bf16_bits(s) if dtype == "bf16" else s.astype(np.float16)
    return {"qweight": qweight, "qzeros": qzeros, "scales": scales}


def make_x(M, K, seed=0, dtype="f16"):
    """Activations [M, K], standard normal: fp16, or (dtype="bf16") bfloat16 bits as uint16."""
    x = _rng(seed, "x", M, K).standard_normal((M, K))
    return bf16_bits(x) if dtype == "bf16" else x.astype(np.float16)


# Layer shapes (K, N) of the pages' model.
SHAPES = {
    "qkv": (2048, 3072),
    "gate_up": (2048, 13312),
    "down": (6656, 2048),
    "square": (2048, 2048),
    "lm_head": (2048, 131072),
    "tail80": (6656, 80),
}
