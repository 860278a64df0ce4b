"""Expert sharding of the layer across GPUs (one process per GPU).

"多卡 CUDA 张量并行：DwarfStar 如何在 8 张 L40S 上跑出 120 t/s", section "8 张卡是怎么
配对的": within a pair of GPUs the routed experts are split 50/50 while the
router is replicated. Here every rank holds the weights of a contiguous range
of experts (``expert_shard``), sees the same activations and router logits,
runs the whole layer over its range (moe_ffn_forward with
expert_lo/expert_hi; the other experts' pairs are dropped in its bucketing),
and the ranks' partial outputs are exchanged (``gather_partials``, one
all-gather) and summed in ascending rank order by the library
(moe_sum_partials), so every rank holds the same bits. torch.distributed is
only the transport; the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

from typing import List, Tuple

import torch

from . import _lib


def expert_shard(n_experts: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous range [lo, hi) of the experts held by `rank` of `world`:
    sizes differ by at most one, lower ranks take the larger shares."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    base, extra = divmod(n_experts, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def gather_partials(partial: torch.Tensor, group=None) -> List[torch.Tensor]:
    """All ranks' partials, in rank order, on the device of `partial` (one
    all-gather). Works over NCCL (CUDA tensors) and gloo (through host
    copies)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    backend = dist.get_backend(group)
    src = partial if (backend == "nccl" or partial.device.type == "cpu") else partial.cpu()
    bufs = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(bufs, src.contiguous(), group=group)
    return [b.to(partial.device, non_blocking=False) for b in bufs]


class ShardedLayer:
    """One rank's share of an expert-sharded layer. `table` holds this rank's
    experts' weights for [lo, hi) (the other experts' entries are never read:
    their pairs are dropped before any weight access). `n_experts` is the
    table length, routed plus shared experts: the shared experts are the last
    entries, so the last rank's range computes them, once."""

    def __init__(self, table, n_experts: int, rank: int, world: int, group=None):
        self.table, self.group = table, group
        self.lo, self.hi = expert_shard(n_experts, rank, world)
        self.n_experts = n_experts

    def forward(self, x_bf16: torch.Tensor, logits: torch.Tensor, k: int, renormalize: bool = True,
                path: int = _lib.PATH_AUTO) -> torch.Tensor:
        opt = _lib.make_options(renormalize=renormalize, expert_lo=self.lo, expert_hi=self.hi,
                                n_experts=self.n_experts, path=path)
        partial = _lib.ffn_forward(self.table, x_bf16, logits, k, options=opt)
        parts = torch.stack(gather_partials(partial, self.group))
        return _lib.sum_partials(parts)
