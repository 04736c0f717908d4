"""qdot_t split across the ranks of a process group (one process per GPU).

Each output column j of qdot_t depends only on weight row W[j, :] and its scales
WS[j, :], and each output row i only on A[i, :] and AS[i, :] ("Quantized
built-ins and formats", section "Q8_0", the qdot_t formula: the sum runs over
the K blocks of one activation row and one weight row).  So the contraction
splits two ways with no exchange inside it:

* column split (N): rank r holds weight rows [n_lo(r), n_hi(r)) and their
  scales, the activation rows are replicated, and each rank computes
  C[:, n_lo:n_hi].  The full C is one all-gather along N, or stays sharded
  for a following column-parallel operation;
* row split (M), for prompt-sized M: rank r takes activation rows
  [m_lo(r), m_hi(r)), the weights are replicated, and the full C is one
  all-gather along M (contiguous in the row-major C).

The local contraction on each rank is the library's own (pq_quantize_qdot_q8_0
or pq_qdot_q8_0_ex on that rank's device memory); only the gather goes through
torch.distributed (NCCL on GPUs).  No kernel ever reads another rank's memory.
Shards are as even as possible: the first N % world ranks take one more row.
The all-gather needs equal sizes, so shorter shards are padded by one row
(column) and the padding is dropped when the gathered result is assembled.
"""
from __future__ import annotations

from typing import Callable

import torch


def shard_range(n: int, world: int, rank: int) -> tuple[int, int]:
    """[lo, hi) of rank `rank` when n items are split over `world` ranks."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"bad split: n={n} world={world} rank={rank}")
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def shard_weights(W: torch.Tensor, WS: torch.Tensor, world: int, rank: int, ws_layout: int = 0):
    """This rank's weight rows and their scales (contiguous): W [n_r, K] and WS [n_r, K/32]
    (ws_layout 0) or [K/32, n_r] (ws_layout 1, the qmma_t layout)."""
    N = W.shape[0]
    lo, hi = shard_range(N, world, rank)
    Wl = W[lo:hi].contiguous()
    WSl = (WS[lo:hi] if ws_layout == 0 else WS[:, lo:hi]).contiguous()
    return Wl, WSl


def _gather_dim(local: torch.Tensor, sizes: list[int], dim: int, group=None) -> torch.Tensor:
    """All-gather of per-rank blocks along `dim` (0: rows, 1: columns) of unequal sizes."""
    import torch.distributed as dist
    world = len(sizes)
    width = max(sizes)
    if local.shape[dim] < width:  # pad to the common size of the collective
        pad_shape = list(local.shape)
        pad_shape[dim] = width - local.shape[dim]
        local = torch.cat([local, local.new_zeros(pad_shape)], dim=dim)
    # the collective concatenates the ranks' blocks along the first dimension
    out = local.new_empty((world * local.shape[0],) + tuple(local.shape[1:]))
    dist.all_gather_into_tensor(out, local.contiguous(), group=group)
    if dim == 0:
        if all(s == width for s in sizes):
            return out
        return torch.cat([out[r * width: r * width + sizes[r]] for r in range(world)], dim=0)
    blocks = out.view(world, local.shape[0], width)
    return torch.cat([blocks[r, :, :sizes[r]] for r in range(world)], dim=1)


class ColumnSplit:
    """qdot_t with the weight rows split over the ranks (N split).

    `W_local`, `WS_local`: this rank's shard (see shard_weights).  `local_qdot`
    computes C_local = qdot_t(A, AS, W_local, WS_local) on this rank's data;
    by default the library's pq_qdot_q8_0_ex.  `local_step` computes the
    one-call decode step (quantize x, then contract) on this rank's data; by
    default pq_quantize_qdot_q8_0.
    """

    def __init__(self, W_local: torch.Tensor, WS_local: torch.Tensor, N: int, world: int, rank: int,
                 ws_layout: int = 0, group=None,
                 local_qdot: Callable | None = None, local_step: Callable | None = None):
        self.N, self.world, self.rank, self.group = N, world, rank, group
        self.ws_layout = ws_layout
        self.sizes = [hi - lo for lo, hi in (shard_range(N, world, r) for r in range(world))]
        if W_local.shape[0] != self.sizes[rank]:
            raise ValueError(f"rank {rank} holds {W_local.shape[0]} weight rows, expected {self.sizes[rank]}")
        self.W, self.WS = W_local, WS_local
        if local_qdot is None or local_step is None:
            from . import binding
            local_qdot = local_qdot or (lambda A, AS, W, WS, layout: binding.qdot_q8_0_ex(
                A, AS, W, WS, ws_layout=layout))
            local_step = local_step or (lambda x, W, WS, layout: binding.quantize_qdot_q8_0(
                x, W, WS, ws_layout=layout))
        self.local_qdot, self.local_step = local_qdot, local_step

    def qdot(self, A: torch.Tensor, AS: torch.Tensor, gather: bool = True) -> torch.Tensor:
        """C = qdot_t(A, AS, W, WS): [M, N] all-gathered, or this rank's [M, n_r] columns."""
        C = self.local_qdot(A, AS, self.W, self.WS, self.ws_layout)
        return _gather_dim(C, self.sizes, 1, self.group) if gather and self.world > 1 else C

    def step(self, x: torch.Tensor, gather: bool = True) -> torch.Tensor:
        """One decode step on the shard (x replicated on every rank), then the gather."""
        C = self.local_step(x, self.W, self.WS, self.ws_layout)
        return _gather_dim(C, self.sizes, 1, self.group) if gather and self.world > 1 else C


class RowSplit:
    """qdot_t with the activation rows split over the ranks (M split; weights replicated)."""

    def __init__(self, W: torch.Tensor, WS: torch.Tensor, world: int, rank: int, ws_layout: int = 0,
                 group=None, local_qdot: Callable | None = None):
        self.W, self.WS, self.world, self.rank, self.group = W, WS, world, rank, group
        self.ws_layout = ws_layout
        if local_qdot is None:
            from . import binding
            local_qdot = lambda A, AS, W, WS, layout: binding.qdot_q8_0_ex(A, AS, W, WS, ws_layout=layout)  # noqa: E731
        self.local_qdot = local_qdot

    def rows(self, M: int) -> tuple[int, int]:
        return shard_range(M, self.world, self.rank)

    def qdot(self, A: torch.Tensor, AS: torch.Tensor, gather: bool = True) -> torch.Tensor:
        """A, AS: the full activation rows (each rank reads its own range).  Returns C [M, N]
        all-gathered, or this rank's rows."""
        M = A.shape[0]
        lo, hi = self.rows(M)
        C = self.local_qdot(A[lo:hi].contiguous(), AS[lo:hi].contiguous(), self.W, self.WS, self.ws_layout)
        if not gather or self.world == 1:
            return C
        sizes = [h - l for l, h in (shard_range(M, self.world, r) for r in range(self.world))]
        return _gather_dim(C, sizes, 0, self.group)
