"""Degenerate and extreme cases of the layer on the GPU, against the oracle:
every slot a sentinel (no live rows: no GEMM tile is issued and every output
row is zero), a single token, one expert with k = 1 (a dense SwiGLU MLP),
every expert picked (k = E), and the largest expert count with k = 8."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import dev, dev_bf16, host, host_bf16_bits, host_f32_from_bf16, require_gpu, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def _forward(moe, wl, fp8=False, mask=None):
    x, W1, W2 = synth.hidden_states(wl), synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    logits = synth.router_logits(wl)
    if fp8:
        q1, s1 = oracle.quant_weight_fp8(W1)
        q2, s2 = oracle.quant_weight_fp8(W2)
        ref = oracle.moe_forward(x, q1, q2, W1_scales=s1, W2_scales=s2, E=wl.E, k=wl.k, logits=logits,
                                 sentinel_mask=mask)
        w1d, w2d, s1d, s2d = dev(q1), dev(q2), dev(s1), dev(s2)
    else:
        ref = oracle.moe_forward(x, W1, W2, E=wl.E, k=wl.k, logits=logits, sentinel_mask=mask)
        w1d, w2d, s1d, s2d = dev_bf16(W1), dev_bf16(W2), None, None
    out = torch.full((wl.T, wl.H), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    a = moe.forward_args(dtype=moe.MOE_FP8_E4M3_B128 if fp8 else moe.MOE_BF16, T=wl.T, E=wl.E, k=wl.k,
                         H=wl.H, I=wl.I, x=dev_bf16(x), W1=w1d, W2=w2d, W1_scales=s1d, W2_scales=s2d, out=out,
                         logits=dev(logits), sentinel_mask=None if mask is None else dev(mask))
    n = moe.moe_forward_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    moe.moe_forward(a, ws, n)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    return host_f32_from_bf16(out), ref


@pytest.mark.parametrize("fp8", [False, True])
def test_every_slot_a_sentinel(moe, fp8):
    wl = synth.Workload("all-sentinel", T=40, E=8, k=2, H=256, I=256)
    mask = np.ones(wl.R, np.uint8)
    y, ref = _forward(moe, wl, fp8, mask)
    assert ref["offsets"][-1] == 0
    assert np.all(ref["out"] == 0) and np.all(y == 0)


def test_grouped_gemm_with_no_live_rows_zero_fills(moe):
    E, M_cap, N, K = 4, 300, 264, 128
    off = np.zeros(E + 1, np.int32)
    A = torch.full((M_cap, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    B = torch.ones((E, N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M_cap, N), 9, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    moe.moe_grouped_gemm(moe.MOE_BF16, A, None, B, None, dev(off), E, M_cap, N, K, moe.MOE_EPI_STORE, C, None)
    assert moe.moe_get_device_error() == 0
    assert np.all(host_bf16_bits(C) == 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_single_token(moe, fp8):
    wl = synth.Workload("one-token", T=1, E=16, k=4, H=256, I=384)
    y, ref = _forward(moe, wl, fp8)
    assert row_rel_err(y, ref["out"]).max() <= (4e-2 if fp8 else 2e-2)


def test_one_expert_is_a_dense_mlp(moe):
    wl = synth.Workload("dense", T=200, E=1, k=1, H=256, I=512)
    y, ref = _forward(moe, wl)
    assert np.all(ref["w"] == 1.0)
    assert row_rel_err(y, ref["out"]).max() <= 2e-2


def test_every_expert_picked(moe):
    wl = synth.Workload("k-equals-e", T=64, E=8, k=8, H=128, I=256)
    y, ref = _forward(moe, wl)
    assert row_rel_err(y, ref["out"]).max() <= 2e-2


def test_largest_expert_count(moe):
    wl = synth.Workload("e256", T=96, E=256, k=8, H=128, I=128, n_sentinel=40)
    y, ref = _forward(moe, wl, mask=synth.sentinel_mask(wl))
    assert row_rel_err(y, ref["out"]).max() <= 2e-2
    y8, ref8 = _forward(moe, wl, fp8=True, mask=synth.sentinel_mask(wl))
    assert row_rel_err(y8, ref8["out"]).max() <= 4e-2
