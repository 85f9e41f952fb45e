"""Expert parallelism on one GPU ("Mixture of Experts in transformers",
section on expert parallelism).  The id remap kernel (moe_ep_local_ids)
against the oracle's, bit for bit; then the recipe of
grouped_gemm_serving_gb300.ep with the library's steps, its ranks run one
after another on this GPU (no collective: the partial outputs are summed
here), against the unsharded layer on the GPU and the oracle.  Only the
all-reduce itself needs several GPUs; its orchestration is tested over gloo
on CPU."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import dev, dev_bf16, host, host_f32_from_bf16, require_gpu, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


@pytest.mark.parametrize("T,k,E,P", [(1, 1, 2, 2), (333, 3, 37, 3), (4096, 8, 256, 4), (5, 7, 7, 7)])
def test_local_ids_bit_exact(moe, T, k, E, P):
    g = np.random.default_rng(T + E)
    ids = g.integers(0, E + 1, size=(T, k)).astype(np.int32)        # includes the global sentinel E
    ids_d = dev(ids)
    for r in range(P):
        first, n = r * E // P, (r + 1) * E // P - r * E // P
        out = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        moe.moe_ep_local_ids(ids_d, T, k, E, first, n, out)
        assert moe.moe_get_device_error() == 0
        assert np.array_equal(host(out), oracle.ep_local_ids(ids, E, first, n))


def test_local_ids_in_place_and_bad_ids(moe):
    T, k, E = 101, 3, 16
    ids = np.random.default_rng(5).integers(0, E + 1, size=(T, k)).astype(np.int32)
    ids[7, 1], ids[50, 2] = -3, E + 4                                  # not expert ids at all
    t = dev(ids)
    moe.moe_ep_local_ids(t, T, k, E, 4, 8, t)                          # same buffer in and out
    assert moe.moe_get_device_error() == moe.MOE_DEVERR_ROUTE
    assert np.array_equal(host(t), oracle.ep_local_ids(ids, E, 4, 8))
    assert host(t)[7, 1] == 8 and host(t)[50, 2] == 8


def _shard_weights(moe, wl, fp8):
    W1, W2 = synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    if not fp8:
        return dev_bf16(W1), dev_bf16(W2), None, None, (W1, W2, None, None)
    q1, s1 = oracle.quant_weight_fp8(W1)
    q2, s2 = oracle.quant_weight_fp8(W2)
    return dev(q1), dev(q2), dev(s1), dev(s2), (q1, q2, s1, s2)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("P", [2, 3])
def test_sharded_layer_sums_to_the_layer(moe, fp8, P):
    from grouped_gemm_serving_gb300.ep import ExpertParallelMoE, expert_shard
    wl = synth.Workload("ep", T=300, E=10, k=3, H=256, I=384, n_sentinel=25, bias="normal0.5",
                        dtype="fp8" if fp8 else "bf16")
    dtype = moe.MOE_FP8_E4M3_B128 if fp8 else moe.MOE_BF16
    W1, W2, S1, S2, host_w = _shard_weights(moe, wl, fp8)
    x, logits, bias, mask = (dev_bf16(synth.hidden_states(wl)), dev(synth.router_logits(wl)),
                             dev(synth.expert_bias(wl)), dev(synth.sentinel_mask(wl)))
    total = torch.zeros((wl.T, wl.H), dtype=torch.float32, device="cuda")
    for r in range(P):
        first, n = expert_shard(wl.E, P, r)
        sl = slice(first, first + n)
        layer = ExpertParallelMoE(E=wl.E, k=wl.k, H=wl.H, I=wl.I, rank=r, world=P, W1=W1[sl], W2=W2[sl],
                                  W1_scales=None if S1 is None else S1[sl],
                                  W2_scales=None if S2 is None else S2[sl], dtype=dtype)
        total += layer.partial(x, logits, bias, mask).float()
        assert moe.moe_get_device_error() == 0
    # the unsharded layer on the GPU
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    a = moe.forward_args(dtype=dtype, T=wl.T, E=wl.E, k=wl.k, H=wl.H, I=wl.I, x=x, W1=W1, W2=W2, W1_scales=S1,
                         W2_scales=S2, out=out, logits=logits, expert_bias=bias, sentinel_mask=mask)
    nws = moe.moe_forward_workspace_size(a)
    moe.moe_forward(a, torch.empty(nws, dtype=torch.uint8, device="cuda"), nws)
    assert moe.moe_get_device_error() == 0
    got, one = host(total), host_f32_from_bf16(out)
    # the ranks' partial outputs are rounded to bf16 before the sum (each by
    # at most 2^-9 of its own size), the unsharded output once
    assert row_rel_err(got, one).max() <= 1e-2
    q1, q2, s1, s2 = host_w
    ref = oracle.moe_forward(synth.hidden_states(wl), q1, q2, W1_scales=s1, W2_scales=s2, E=wl.E, k=wl.k,
                             logits=synth.router_logits(wl), bias=synth.expert_bias(wl),
                             sentinel_mask=synth.sentinel_mask(wl))["out"]
    assert row_rel_err(got, ref).max() <= (4e-2 if fp8 else 2e-2)
