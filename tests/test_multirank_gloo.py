"""The multi-rank paths on CPU, world size 2 over gloo (127.0.0.1).

1. bench.py's replica aggregation: every rank times its own batch; the job's
   time is the slowest rank's (max over ranks) and its throughput counts every
   rank's tokens.
2. Expert parallelism as "Mixture of Experts in transformers" describes it
   (section on expert parallelism): each rank holds E/2 experts (weights
   sharded on the expert dimension), remaps global expert ids to local ones,
   turns picks of non-local experts into sentinels, runs its local layer, and
   an all-reduce sums the partial outputs.  The sum must equal the unsharded
   layer.  The per-rank layer is the oracle here (CPU only)."""
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


def _ep_ranks(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from grouped_gemm_serving_gb300 import synth
    _init(rank, world, port)
    try:
        wl = synth.Workload("ep", T=48, E=8, k=2, H=128, I=128, n_sentinel=6)
        x = synth.hidden_states(wl)
        ids, w = oracle.route_topk(synth.router_logits(wl), None, wl.k)
        ids = oracle.mark_sentinels(ids, synth.sentinel_mask(wl), wl.E)
        E_loc = wl.E // world
        lo = rank * E_loc                         # this rank's experts [lo, lo + E_loc)
        local = (ids >= lo) & (ids < lo + E_loc)
        ids_loc = np.where(local, ids - lo, E_loc).astype(np.int32)   # others -> sentinel
        experts = list(range(lo, lo + E_loc))
        W1 = synth.expert_weights(wl, "w1", experts=experts)
        W2 = synth.expert_weights(wl, "w2", experts=experts)
        part = oracle.moe_forward(x, W1, W2, E=E_loc, k=wl.k, ids=ids_loc, w=w)["out"]
        t = torch.from_numpy(part.astype(np.float64))
        dist.all_reduce(t)                        # sum of the partial outputs
        out[rank] = t.numpy()
    finally:
        dist.destroy_process_group()


def test_expert_parallel_partials_sum_to_the_full_layer():
    import oracle
    from grouped_gemm_serving_gb300 import synth
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_ep_ranks, args=(2, port, out), nprocs=2, join=True)
    wl = synth.Workload("ep", T=48, E=8, k=2, H=128, I=128, n_sentinel=6)
    full = oracle.moe_forward(synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                              synth.expert_weights(wl, "w2"), E=wl.E, k=wl.k,
                              logits=synth.router_logits(wl), sentinel_mask=synth.sentinel_mask(wl))
    assert np.array_equal(out[0], out[1])
    np.testing.assert_allclose(out[0], full["out"], rtol=1e-5, atol=1e-6)
    dead = (full["ids"] == wl.E).all(axis=1)
    assert np.all(out[0][dead] == 0)
