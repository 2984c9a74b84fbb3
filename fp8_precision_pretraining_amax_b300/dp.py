"""Data-parallel sharding of the block-scaled FP8 linear layer over tokens.

The pages train with data parallelism (the Puro-2B report, section 1: DP and
PP across RTX 5090 nodes, gradients all-reduced over PCIe P2P / GPUDirect
RDMA).  For one linear layer that means: each rank holds a shard of the
tokens; Fprop and Dgrad of a shard need nothing from other ranks (their
outputs are rows of the full outputs); Wgrad sums over all tokens, so each
rank computes the FP32 Wgrad of its shard and the ranks add them with one
all-reduce -- the only exchange on this path.

This module is host-side logic only: the shard boundaries, the all-reduce,
and `LinearFP8DP`, which strings the library's launches together for one
rank.  Shards are whole 128-token blocks (the column-wise tiles that Wgrad
reduces over never straddle ranks).
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist

BLOCK = 128


def token_shard(M: int, rank: int, world: int) -> Tuple[int, int]:
    """[m0, m1) of the tokens rank `rank` of `world` owns: consecutive runs of
    whole 128-token blocks, block counts differing by at most one between
    ranks (the first M/128 % world ranks get one more)."""
    if M % BLOCK:
        raise ValueError(f"token count {M} is not a multiple of {BLOCK}")
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world of {world}")
    blocks = M // BLOCK
    base, extra = divmod(blocks, world)
    b0 = rank * base + min(rank, extra)
    b1 = b0 + base + (1 if rank < extra else 0)
    return b0 * BLOCK, b1 * BLOCK


def allreduce_wgrad_(dw: torch.Tensor, group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """Sum the per-rank Wgrad partials in place (every rank gets the sum)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dw, op=dist.ReduceOp.SUM, group=group)
    return dw


class LinearFP8DP:
    """One rank's part of a data-parallel step of an nn.Linear on the FP8 path.

    The rank holds `M_local` tokens (its shard); the weight is replicated.
    step() quantizes, runs Fprop and Dgrad on the shard, computes the shard's
    Wgrad in FP32 and all-reduces it, so `dw` holds the Wgrad of all tokens
    on every rank."""

    def __init__(self, M_local: int, K: int, N: int, device="cuda", group=None):
        from .linear import LinearFP8
        self.layer = LinearFP8(M_local, K, N, device=device)
        self.dw = torch.empty((N, K), dtype=torch.float32, device=device)
        self.group = group

    def step(self, x: torch.Tensor, w: torch.Tensor, dy: torch.Tensor):
        from . import fp8bq
        L = self.layer
        L.forward(x, w)
        fp8bq.fp8bq_quantize_rowcol(dy, L.dyq, L.sdy, L.dyqT, L.sdyT)
        fp8bq.fp8bq_gemm_dgrad(L.dyq, L.sdy, L.wqT, L.sw, L.dx)
        fp8bq.fp8bq_gemm_wgrad_f32(L.dyqT, L.sdyT, L.xqT, L.sxT, self.dw)
        allreduce_wgrad_(self.dw, self.group)
        return L.y, L.dx, self.dw
