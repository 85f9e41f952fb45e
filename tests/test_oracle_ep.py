"""Pins of the oracle's expert-parallel id remap ("Mixture of Experts in
transformers", expert parallelism: experts sharded on their first dimension,
global router ids remapped to local ones, non-local picks left out).

- Partition: over the ranks of any sharding, every live global pick is live
  on exactly one rank, and first + local id gives the global id back; the
  global sentinel (and any id outside [0, E]) is a sentinel on every rank.
- Partial sums: the layer of each rank on its local ids and its own experts'
  weights, summed over the ranks, is the unsharded layer (the linear combine
  splits over the experts), with and without sentinels, bf16 and FP8."""
import numpy as np
import pytest

import oracle
from grouped_gemm_serving_gb300 import synth


def _shards(E, P):
    return [(r * E // P, (r + 1) * E // P - r * E // P) for r in range(P)]


@pytest.mark.parametrize("E,P", [(8, 2), (256, 4), (10, 3), (5, 5), (7, 1)])
def test_every_pick_is_local_on_exactly_one_rank(E, P):
    g = np.random.default_rng(E * 31 + P)
    ids = g.integers(-2, E + 3, size=4000).astype(np.int32)       # includes E and bad ids
    live_on = np.zeros(ids.size, np.int64)
    back = np.full(ids.size, -1, np.int64)
    for first, n in _shards(E, P):
        loc = oracle.ep_local_ids(ids, E, first, n)
        assert loc.dtype == np.int32 and np.all((loc >= 0) & (loc <= n))
        live = loc < n
        live_on += live
        back[live] = first + loc[live]
    valid = (ids >= 0) & (ids < E)
    assert np.all(live_on[valid] == 1) and np.all(live_on[~valid] == 0)
    assert np.array_equal(back[valid], ids[valid])


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("P", [2, 3])
def test_rank_partials_sum_to_the_layer(fp8, P):
    wl = synth.Workload("ep", T=40, E=9, k=3, H=128, I=256, n_sentinel=7, bias="normal0.5",
                        dtype="fp8" if fp8 else "bf16")
    x, W1, W2 = (synth.hidden_states(wl), synth.expert_weights(wl, "w1"),
                 synth.expert_weights(wl, "w2"))
    s1 = s2 = None
    if fp8:
        W1, s1 = oracle.quant_weight_fp8(W1)
        W2, s2 = oracle.quant_weight_fp8(W2)
    full = oracle.moe_forward(x, W1, W2, W1_scales=s1, W2_scales=s2, E=wl.E, k=wl.k,
                              logits=synth.router_logits(wl), bias=synth.expert_bias(wl),
                              sentinel_mask=synth.sentinel_mask(wl))
    total = np.zeros_like(full["out"], dtype=np.float64)
    for first, n in _shards(wl.E, P):
        loc = oracle.ep_local_ids(full["ids"], wl.E, first, n)
        sl = slice(first, first + n)
        part = oracle.moe_forward(x, W1[sl], W2[sl], W1_scales=None if s1 is None else s1[sl],
                                  W2_scales=None if s2 is None else s2[sl], E=n, k=wl.k, ids=loc, w=full["w"])
        assert part["offsets"][-1] == int((loc < n).sum())
        total += part["out"]
    np.testing.assert_allclose(total, full["out"], rtol=1e-5, atol=1e-6)
    dead = (full["ids"] == wl.E).all(axis=1)
    assert np.all(total[dead] == 0)
