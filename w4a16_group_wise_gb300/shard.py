"""Column-parallel (N-sharded) use of the W4A16 layer across ranks.

"Carga de capas cuantizadas: AWQ / GPTQ / Marlin / fp8" (sections "Motivacion de diseno" and
"Limites y fallos") describes quantized linears split across tensor-parallel ranks: a
column-parallel layer shards the output dimension, and its scales are split with it.  Output
columns are independent (y[:, n] needs only column n of W), so each rank repacks and multiplies
only its own range of columns and no collective is needed on the data path; the slices of y are
gathered only when a consumer wants y whole.

Slices start on 64-column boundaries (the packed layout's n-blocks), so each rank's slice is a
layer of its own: w4a16_repack_chunk reads it straight out of the full AWQ tensors (their row
strides), and the ragged remainder of N goes to the last rank.
"""
import torch

from . import binding

BLOCK_N = 64  # columns per n-block of the packed layout


def column_slices(N, world):
    """The column ranges [(n0, n1), ...] of ranks 0 .. world-1: contiguous, covering [0, N), each
    start a multiple of 64, the n-blocks dealt as evenly as possible.  The last ranks take the extra
    n-blocks, so the last rank, which holds the ragged last n-block, is never short by more than
    that block's missing columns: widths differ by at most 64.  When there are fewer n-blocks than
    ranks, the first ranks get empty ranges (n0 == n1 == 0)."""
    if N <= 0 or world <= 0:
        raise ValueError("N and world must be positive")
    nb = (N + BLOCK_N - 1) // BLOCK_N
    base, extra = divmod(nb, world)
    out, b = [], 0
    for r in range(world):
        cnt = base + (1 if r >= world - extra else 0)
        out.append((min(BLOCK_N * b, N), min(BLOCK_N * (b + cnt), N)))
        b += cnt
    return out


def repack_slice(qweight, qzeros, scales, K, N, g, n0, n1, stream=None):
    """The packed buffer of columns [n0, n1) of a K x N layer, as a layer of its own (K x (n1 - n0)),
    read from the full AWQ tensors (qweight int32 [K, N/8], qzeros int32 [K/g, N/8], scales
    [K/g, N]) without copying them."""
    if n0 % BLOCK_N or not (0 <= n0 < n1 <= N) or (n1 % 8):
        raise ValueError("slice [%d, %d) of %d columns: start a multiple of 64, end a multiple of 8" % (n0, n1, N))
    ns = n1 - n0
    packed = torch.empty(binding.packed_bytes(K, ns, g), dtype=torch.uint8, device=qweight.device)
    binding.repack_chunk(qweight[:, n0 // 8:n1 // 8], qzeros[:, n0 // 8:n1 // 8], scales[:, n0:n1], K, ns, g, 0, ns,
                         packed, stream=stream)
    return packed


class ColumnParallelLinear:
    """One rank's share of a column-parallel W4A16 linear: columns [n0, n1) of the layer."""

    def __init__(self, qweight, qzeros, scales, K, N, g, rank, world, stream=None):
        self.K, self.N, self.g = K, N, g
        self.rank, self.world = rank, world
        self.slices = column_slices(N, world)
        self.n0, self.n1 = self.slices[rank]
        self.width = self.n1 - self.n0
        self.packed = (repack_slice(qweight, qzeros, scales, K, N, g, self.n0, self.n1, stream)
                       if self.width else None)

    def forward(self, x, y=None, workspace=None, stream=None):
        """This rank's columns of y = x . W: [M, n1 - n0], in x's element type."""
        M = x.shape[0]
        if self.width == 0:
            return torch.empty((M, 0), dtype=x.dtype, device=x.device)
        return binding.gemm(x, self.packed, M, self.width, self.K, self.g, y=y, workspace=workspace, stream=stream)

    def gather(self, y_local, group=None):
        """The whole y [M, N] from every rank's columns (an all-gather over torch.distributed; the
        slices are padded to the widest and trimmed back)."""
        import torch.distributed as dist
        widest = max(n1 - n0 for n0, n1 in self.slices)
        M = y_local.shape[0]
        pad = torch.zeros((M, widest), dtype=y_local.dtype, device=y_local.device)
        pad[:, :y_local.shape[1]] = y_local
        parts = [torch.empty_like(pad) for _ in range(self.world)]
        dist.all_gather(parts, pad.contiguous(), group=group)
        return torch.cat([p[:, :n1 - n0] for p, (n0, n1) in zip(parts, self.slices)], dim=1)
