"""The weighted combine folded into the down GEMM (moe_grouped_gemm_combine,
moe_forward's MOE_FWD_FUSED_COMBINE): bit for bit the results of
moe_grouped_gemm + moe_combine, whichever CTA stores a token's last row --
over top-k 1 to 8, sentinel slots and tokens with only sentinels, feature
counts that end in a partial 128-feature block, and calls in a row (the
counters reset themselves)."""
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


CASES = [
    # T, E, k, H, I, sentinel slots
    (300, 16, 4, 256, 384, 40),
    (97, 12, 3, 200, 136, 5),
    (64, 8, 2, 128, 256, 8),
    (1000, 32, 8, 2880, 256, 300),
    (50, 1, 1, 384, 128, 3),
    (2048, 64, 8, 1024, 128, 0),
]


def _layer(moe, T, E, k, H, I, n_sent, seed):
    wl = synth.Workload("fc", T=T, E=E, k=k, H=H, I=I, n_sentinel=n_sent, bias="normal0.5", seed=seed)
    ids, w = oracle.route_topk(synth.router_logits(wl), synth.expert_bias(wl), k)
    mask = synth.sentinel_mask(wl)
    if mask is not None:
        ids = oracle.mark_sentinels(ids, mask, E)
    if T >= 50:
        ids[7] = E                                           # a token with only sentinel slots
    r = moe.route_sort_t(E, k, topk_ids=dev(ids))
    R = T * k
    h = dev_bf16(synth.dense_rows(R, I, seed, std=1.0))
    W2 = dev_bf16(synth.expert_weights(wl, "w2"))
    return wl, ids, dev(w), r, h, W2


@pytest.mark.parametrize("T,E,k,H,I,n_sent", CASES)
def test_equals_gemm_then_combine(moe, T, E, k, H, I, n_sent):
    wl, ids, w, r, h, W2 = _layer(moe, T, E, k, H, I, n_sent, seed=T + H)
    R = T * k
    ids_d = r["ids"]
    y_ref = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
    out_ref = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm(moe.MOE_BF16, h, None, W2, None, r["offsets"], E, R, H, I, moe.MOE_EPI_STORE, y_ref, None)
    moe.moe_combine(y_ref, ids_d, w, r["row_pos"], T, k, H, E, out_ref)
    nws = moe.moe_grouped_gemm_combine_workspace_size(T, H)
    ws = torch.full((nws,), 0xAB, dtype=torch.uint8, device="cuda")   # garbage: the call clears its counters
    for _ in range(2):                                                  # calls in a row
        y = torch.full((R, H), 5, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        out = torch.full((T, H), 5, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        moe.moe_grouped_gemm_combine(h, W2, r["offsets"], E, R, H, I, ids_d, w, r["sorted_rows"], r["row_pos"], T, k,
                                     y, out, ws, nws)
        assert moe.moe_get_device_error() == 0
        assert np.array_equal(host_bf16_bits(y), host_bf16_bits(y_ref))
        assert np.array_equal(host_bf16_bits(out), host_bf16_bits(out_ref))
    if T >= 50:
        assert np.all(host_bf16_bits(out)[7] == 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_forward_flag(moe, fp8):
    wl = synth.Workload("fc-fwd", T=400, E=16, k=4, H=256, I=384, n_sentinel=50, bias="normal0.5",
                        dtype="fp8" if fp8 else "bf16")
    x, W1, W2 = synth.hidden_states(wl), synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    logits, mask = synth.router_logits(wl), synth.sentinel_mask(wl)
    s1 = s2 = None
    if fp8:
        W1, s1 = oracle.quant_weight_fp8(W1)
        W2, s2 = oracle.quant_weight_fp8(W2)
        wd1, wd2 = dev(W1), dev(W2)
    else:
        wd1, wd2 = dev_bf16(W1), dev_bf16(W2)
    outs = []
    for fused in (False, True):
        out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
        a = moe.forward_args(dtype=moe.MOE_FP8_E4M3_B128 if fp8 else moe.MOE_BF16, T=wl.T, E=wl.E, k=wl.k, H=wl.H,
                             I=wl.I, x=dev_bf16(x), W1=wd1, W2=wd2, W1_scales=None if s1 is None else dev(s1),
                             W2_scales=None if s2 is None else dev(s2), out=out, logits=dev(logits),
                             sentinel_mask=dev(mask), fused_combine=fused)
        n = moe.moe_forward_workspace_size(a)
        moe.moe_forward(a, torch.empty(n, dtype=torch.uint8, device="cuda"), n)
        assert moe.moe_get_device_error() == 0
        outs.append(host_bf16_bits(out))
    assert np.array_equal(outs[0], outs[1])
    ref = oracle.moe_forward(x, W1, W2, W1_scales=s1, W2_scales=s2, E=wl.E, k=wl.k, logits=logits,
                             sentinel_mask=mask)["out"]
    got = host_f32_from_bf16(torch.from_numpy(outs[1].view(np.int16)).view(torch.bfloat16))
    assert row_rel_err(got, ref).max() <= (4e-2 if fp8 else 2e-2)
