"""Expert parallelism for the MoE layer, as "Mixture of Experts in
transformers" describes it (section on expert parallelism): the stacked
expert weights are sharded on their first dimension (GroupedGemmParallel),
every rank runs the same router over all E experts, remaps the global expert
ids to its local ones with the picks of other ranks' experts masked
(RouterParallel), runs its local layer, and an all-reduce sums the partial
outputs.  The masked picks are sentinels to the local layer (section 2 of the
transformers MoE/FP8 write-up): left out of its histogram, sort and GEMMs and
skipped by its combine, so each rank computes only its own experts' share.

The recipe is written over a small set of steps (``LibraryOps``): routing,
the id remap and the local layer are calls of the C library on the rank's
GPU; the sum is one ``torch.distributed`` all-reduce of the ``[T, H]``
partial output.  No arithmetic happens here.  Each rank's partial output is
stored in bf16 by the combine before the sum.

Usage, one process per GPU::

    first, n = expert_shard(E, world, rank)
    layer = ExpertParallelMoE(E=E, k=k, H=H, I=I, rank=rank, world=world,
                              W1=W1[first:first + n], W2=W2[first:first + n])
    out = layer.forward(x, logits)          # the full layer's output on every rank

No TMA multicast or peer memory is used: every kernel reads its own GPU's
memory, and the only exchange is the all-reduce.
"""
from __future__ import annotations

import torch

from . import moe


def expert_shard(E: int, world: int, rank: int) -> tuple[int, int]:
    """First global expert and number of experts held by `rank` when E
    experts are split in contiguous runs over `world` ranks: rank r holds
    [r*E//world, (r+1)*E//world), so the run lengths differ by at most one."""
    if not (0 <= rank < world) or world > E:
        raise ValueError(f"cannot shard {E} experts over {world} ranks (rank {rank})")
    first = rank * E // world
    return first, (rank + 1) * E // world - first


class LibraryOps:
    """The recipe's steps on this rank's GPU: the library's routing, id remap
    and layer, and an all-reduce of torch.distributed."""

    def __init__(self):
        self._ws = None

    def route(self, logits, expert_bias, sentinel_mask, E, k, renormalize):
        r = moe.route_sort_t(E, k, logits=logits, expert_bias=expert_bias, sentinel_mask=sentinel_mask,
                             renormalize=renormalize)
        return r["ids"], r["w"]

    def local_ids(self, ids, E_global, first, E_local):
        T, k = ids.shape
        out = torch.empty_like(ids)
        moe.moe_ep_local_ids(ids, T, k, E_global, first, E_local, out)
        return out

    def local_layer(self, x, local_ids, w, *, dtype, E_local, H, I, W1, W2, W1_scales, W2_scales):
        T, k = local_ids.shape
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
        a = moe.forward_args(dtype=dtype, T=T, E=E_local, k=k, H=H, I=I, x=x, W1=W1, W2=W2,
                             W1_scales=W1_scales, W2_scales=W2_scales, out=out, topk_ids=local_ids, topk_w=w)
        n = moe.moe_forward_workspace_size(a)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(n, dtype=torch.uint8, device=x.device)
        moe.moe_forward(a, self._ws, n)
        return out

    def all_reduce(self, t, group):
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
        return t


class ExpertParallelMoE:
    """One rank's share of an expert-parallel MoE layer.

    W1 ``[n, 2I, H]`` and W2 ``[n, H, I]`` (with their FP8 block scales) are
    this rank's experts ``[first, first + n)`` of ``expert_shard(E, world,
    rank)``.  ``forward`` takes the full batch (x ``[T, H]`` bf16, router
    logits ``[T, E]`` fp32) on every rank and returns the full layer's output
    on every rank.  With world == 1 the all-reduce is skipped."""

    def __init__(self, *, E, k, H, I, rank, world, W1, W2, W1_scales=None, W2_scales=None,
                 dtype=moe.MOE_BF16, renormalize=True, group=None, ops=None):
        self.E, self.k, self.H, self.I = E, k, H, I
        self.rank, self.world, self.group = rank, world, group
        self.first, self.E_local = expert_shard(E, world, rank)
        if W1.shape[0] != self.E_local or W2.shape[0] != self.E_local:
            raise ValueError(f"rank {rank} holds {self.E_local} experts; got weight stacks of "
                             f"{W1.shape[0]} and {W2.shape[0]}")
        self.W1, self.W2, self.W1_scales, self.W2_scales = W1, W2, W1_scales, W2_scales
        self.dtype, self.renormalize = dtype, renormalize
        self.ops = ops if ops is not None else LibraryOps()

    def partial(self, x, logits, expert_bias=None, sentinel_mask=None):
        """This rank's partial output: the layer over its own experts only."""
        ids, w = self.ops.route(logits, expert_bias, sentinel_mask, self.E, self.k, self.renormalize)
        local = self.ops.local_ids(ids, self.E, self.first, self.E_local)
        return self.ops.local_layer(x, local, w, dtype=self.dtype, E_local=self.E_local, H=self.H, I=self.I,
                                    W1=self.W1, W2=self.W2, W1_scales=self.W1_scales, W2_scales=self.W2_scales)

    def forward(self, x, logits, expert_bias=None, sentinel_mask=None):
        out = self.partial(x, logits, expert_bias, sentinel_mask)
        if self.world > 1:
            out = self.ops.all_reduce(out, self.group)
        return out
