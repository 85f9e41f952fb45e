"""The multi-rank paths on CPU, world sizes 2 and 3 over gloo (127.0.0.1).

1. bench.py's replica aggregation: every rank times its own batch; the job's
   time is the slowest rank's (max over ranks) and its throughput counts every
   rank's tokens.
2. Expert parallelism as "Mixture of Experts in transformers" describes it
   (section on expert parallelism), through the library's recipe
   (grouped_gemm_serving_gb300.ep.ExpertParallelMoE): each rank holds a run of
   the experts (weights sharded on the expert dimension), remaps global
   expert ids to local ones, turns picks of non-local experts into sentinels,
   runs its local layer, and an all-reduce sums the partial outputs.  The sum
   must equal the unsharded layer.  The oracle stands in for the library's
   steps here (CPU only); the GPU tests run the library's steps."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _bench_ranks(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    _init(rank, world, port)
    try:
        ms = [0.75, 0.9][rank]                      # rank 1 is the slow one
        ms_max = bench.cross_rank_max(ms, dist, "cpu")
        val = bench.job_tokens_per_s(4096, world, ms_max)
        out[rank] = (ms_max, val)
    finally:
        dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_bench_ranks, args=(2, port, out), nprocs=2, join=True)
    for r in (0, 1):
        ms_max, val = out[r]
        assert ms_max == 0.9
        assert val == pytest.approx(2 * 4096 / 0.9e-3)


class _OracleOps:
    """The expert-parallel recipe's steps on CPU tensors: the oracle's routing,
    id remap and layer in place of the library's, and the gloo all-reduce."""

    def __init__(self, wl):
        self.wl = wl

    def route(self, logits, expert_bias, sentinel_mask, E, k, renormalize):
        import oracle
        ids, w = oracle.route_topk(logits.numpy(), None if expert_bias is None else expert_bias.numpy(), k,
                                   renormalize)
        if sentinel_mask is not None:
            ids = oracle.mark_sentinels(ids, sentinel_mask.numpy(), E)
        return torch.from_numpy(ids), torch.from_numpy(w)

    def local_ids(self, ids, E_global, first, E_local):
        import oracle
        return torch.from_numpy(oracle.ep_local_ids(ids.numpy(), E_global, first, E_local))

    def local_layer(self, x, local_ids, w, *, dtype, E_local, H, I, W1, W2, W1_scales, W2_scales):
        import oracle
        r = oracle.moe_forward(x.numpy(), W1.numpy(), W2.numpy(), E=E_local, k=local_ids.shape[1],
                               ids=local_ids.numpy(), w=w.numpy())
        return torch.from_numpy(r["out"].astype(np.float64))

    def all_reduce(self, t, group):
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
        return t


EP_WL = dict(T=48, E=9, k=2, H=128, I=128, n_sentinel=6, bias="normal0.5")


def _ep_ranks(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    from grouped_gemm_serving_gb300 import synth
    from grouped_gemm_serving_gb300.ep import ExpertParallelMoE, expert_shard
    _init(rank, world, port)
    try:
        wl = synth.Workload("ep", **EP_WL)
        first, n = expert_shard(wl.E, world, rank)
        experts = list(range(first, first + n))
        layer = ExpertParallelMoE(E=wl.E, k=wl.k, H=wl.H, I=wl.I, rank=rank, world=world,
                                  W1=torch.from_numpy(synth.expert_weights(wl, "w1", experts=experts)),
                                  W2=torch.from_numpy(synth.expert_weights(wl, "w2", experts=experts)),
                                  ops=_OracleOps(wl))
        part = layer.partial(torch.from_numpy(synth.hidden_states(wl)), torch.from_numpy(synth.router_logits(wl)),
                             torch.from_numpy(synth.expert_bias(wl)), torch.from_numpy(synth.sentinel_mask(wl)))
        full = layer.ops.all_reduce(part.clone(), None)
        out[rank] = (first, n, part.numpy(), full.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_partials_sum_to_the_full_layer(world):
    """ExpertParallelMoE's orchestration over gloo ranks (9 experts: uneven
    shards for 2 ranks), with the oracle standing in for the library."""
    import oracle
    from grouped_gemm_serving_gb300 import synth
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_ep_ranks, args=(world, port, out), nprocs=world, join=True)
    wl = synth.Workload("ep", **EP_WL)
    full = oracle.moe_forward(synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                              synth.expert_weights(wl, "w2"), E=wl.E, k=wl.k,
                              logits=synth.router_logits(wl), bias=synth.expert_bias(wl),
                              sentinel_mask=synth.sentinel_mask(wl))
    # the shards tile the experts, and every rank ends with the same sum
    assert sorted((out[r][0], out[r][1]) for r in range(world))[0][0] == 0
    assert sum(out[r][1] for r in range(world)) == wl.E
    for r in range(1, world):
        assert np.array_equal(out[r][3], out[0][3])
    np.testing.assert_allclose(out[0][3], full["out"], rtol=1e-5, atol=1e-6)
    # each rank's partial holds only its own experts' share: nonzero partials
    # are spread over the ranks, and no single rank carries the whole layer
    assert all(np.abs(out[r][2]).max() > 0 for r in range(world))
    assert all(not np.allclose(out[r][2], full["out"]) for r in range(world))
    dead = (full["ids"] == wl.E).all(axis=1)
    assert np.all(out[0][3][dead] == 0)
