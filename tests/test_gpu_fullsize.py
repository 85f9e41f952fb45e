"""Full-size parity: every layer workload at its real size, run through
moe_forward exactly as bench.py launches it, checked against the oracle
on all routing outputs (bit-exact) and on sampled tokens (the oracle computes
those tokens one by one; a token's output depends only on its own row).
Also the live-row sweep of the grouped GEMMs (16384 permuted rows, 128
experts, 100 % / 50 % / 12.5 % live): sampled rows against the oracle and every
sentinel row exactly zero although its input is NaN."""
import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import (dev, dev_bf16, host, host_bf16_bits, host_f32_from_bf16,
                               require_gpu, row_rel_err)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE = {"32e-top4-h2880": 16, "128e-top8-h2048-zipf": 16, "256e-top8-h7168-fp8": 4,
          # decode-sized batches of the same layers (64 tokens)
          "32e-top4-h2880-t64": 16, "256e-top8-h7168-fp8-t64": 4}


@pytest.fixture(scope="module")
def moe():
    require_gpu()
    from grouped_gemm_serving_gb300 import moe as m
    return m


def _device_weights(moe, wl):
    if wl.dtype != "fp8":
        return (dev_bf16(synth.expert_weights(wl, "w1")), dev_bf16(synth.expert_weights(wl, "w2")),
                None, None)
    out = []
    for which, (n, kdim) in (("w1", (2 * wl.I, wl.H)), ("w2", (wl.H, wl.I))):
        q = torch.empty((wl.E, n, kdim), dtype=torch.uint8, device="cuda")
        s = torch.empty((wl.E, (n + 127) // 128, kdim // 128), dtype=torch.float32, device="cuda")
        for e0 in range(0, wl.E, 16):
            ex = list(range(e0, min(wl.E, e0 + 16)))
            wb = dev_bf16(synth.expert_weights(wl, which, experts=ex))
            moe.moe_weight_quant_fp8(wb, len(ex), n, kdim, q[e0:e0 + len(ex)], s[e0:e0 + len(ex)])
            torch.cuda.synchronize()
            del wb
        out += [q, s]
    return out[0], out[2], out[1], out[3]


@pytest.mark.parametrize("name", list(SAMPLE))
def test_full_size_layer(moe, name):
    wl = synth.WORKLOADS[name]
    fp8 = wl.dtype == "fp8"
    x, logits, bias = synth.hidden_states(wl), synth.router_logits(wl), synth.expert_bias(wl)
    W1, W2, S1, S2 = _device_weights(moe, wl)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    ids_d = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w_d = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    a = moe.forward_args(dtype=moe.MOE_FP8_E4M3_B128 if fp8 else moe.MOE_BF16, T=wl.T, E=wl.E, k=wl.k,
                         H=wl.H, I=wl.I, x=dev_bf16(x), W1=W1, W2=W2, W1_scales=S1, W2_scales=S2, out=out,
                         logits=dev(logits), expert_bias=None if bias is None else dev(bias),
                         topk_ids=ids_d, topk_w=w_d, renormalize=wl.renormalize)
    n = moe.moe_forward_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    moe.moe_forward(a, ws, n)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0

    # routing of every token, bit-exact
    ids, w = oracle.route_topk(logits, bias, wl.k, wl.renormalize)
    assert np.array_equal(host(ids_d), ids)
    np.testing.assert_allclose(host(w_d), w, rtol=2e-6)

    # sampled tokens through the oracle, with only the experts they use
    g = np.random.default_rng(123)
    S = np.sort(g.choice(wl.T, SAMPLE[name], replace=False))
    used = np.unique(ids[S])
    remap = np.full(wl.E + 1, -1, np.int64)
    remap[used] = np.arange(used.size)
    ids_c = remap[ids[S]].astype(np.int32)
    W1h = synth.expert_weights(wl, "w1", experts=used)
    W2h = synth.expert_weights(wl, "w2", experts=used)
    kw = dict(E=int(used.size), k=wl.k, ids=ids_c, w=w[S])
    if fp8:
        q1, s1 = oracle.quant_weight_fp8(W1h)
        q2, s2 = oracle.quant_weight_fp8(W2h)
        e0 = int(used[0])                                    # the library's weight quantiser agrees
        assert np.array_equal(host(W1[e0]), q1[0]) and np.array_equal(host(S2[e0]), s2[0])
        ref = oracle.moe_forward(x[S], q1, q2, W1_scales=s1, W2_scales=s2, **kw)["out"]
        tol = 4e-2
    else:
        ref = oracle.moe_forward(x[S], W1h, W2h, **kw)["out"]
        tol = 2e-2
    got = host_f32_from_bf16(out)[S]
    err = row_rel_err(got, ref)
    assert err.max() <= tol, (name, err.max())


@pytest.mark.parametrize("live", [16384, 8192, 2048])
def test_live_row_sweep(moe, live):
    sw = synth.Sweep(live=live)
    wl = sw.workload
    A = synth.sweep_rows(sw)                                 # rows >= live are NaN
    off = synth.sweep_offsets(sw)
    W1 = synth.expert_weights(wl, "w1")
    W2 = synth.expert_weights(wl, "w2")
    M, E, H, I = sw.M_cap, sw.E, sw.H, sw.I
    h = torch.full((M, I), 3, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    y2 = torch.full((M, H), 3, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    offd = dev(off)
    moe.moe_grouped_gemm(moe.MOE_BF16, dev_bf16(A), None, dev_bf16(W1), None, offd, E, M, 2 * I, H,
                         moe.MOE_EPI_SWIGLU, h, None)
    moe.moe_grouped_gemm(moe.MOE_BF16, h, None, dev_bf16(W2), None, offd, E, M, H, I, moe.MOE_EPI_STORE, y2,
                         None)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    assert np.all(host_bf16_bits(h)[live:] == 0)
    assert np.all(host_bf16_bits(y2)[live:] == 0)
    rows = np.sort(np.random.default_rng(live).choice(live, 48, replace=False)).astype(np.int32)
    rows[0], rows[-1] = 0, live - 1
    ref_h = oracle.swiglu(oracle.grouped_gemm_bf16(A, W1, off, rows=rows), len(rows))
    got_h = host_f32_from_bf16(h)[rows]
    assert row_rel_err(got_h, ref_h).max() <= 2e-2
    # the down GEMM on the oracle's own h (rounded to bf16 as the layer stores it)
    hb = np.zeros((M, I), np.uint16)
    hb[rows] = oracle.bf16_round(ref_h)
    ref_y = oracle.grouped_gemm_bf16(hb, W2, off, rows=rows)
    got_y = host_f32_from_bf16(y2)[rows]
    assert row_rel_err(got_y, ref_y).max() <= 2e-2


def test_many_rows_with_sentinels(moe):
    """Two million routed slots (T = 262144 tokens, top-8 of 64 experts) with
    sentinel slots: 2048 sort blocks, row indices in the millions through the
    permute, both GEMMs and the combine.  Routing of every token is checked
    bit-exactly, the layer output on sampled tokens against the oracle."""
    wl = synth.Workload("many-rows", T=262144, E=64, k=8, H=128, I=128, n_sentinel=5000, bias="normal0.5")
    x, logits, bias = synth.hidden_states(wl), synth.router_logits(wl), synth.expert_bias(wl)
    mask = synth.sentinel_mask(wl)
    W1, W2 = synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    ids_d = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w_d = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    a = moe.forward_args(dtype=moe.MOE_BF16, T=wl.T, E=wl.E, k=wl.k, H=wl.H, I=wl.I, x=dev_bf16(x),
                         W1=dev_bf16(W1), W2=dev_bf16(W2), out=out, logits=dev(logits), expert_bias=dev(bias),
                         sentinel_mask=dev(mask), topk_ids=ids_d, topk_w=w_d, renormalize=wl.renormalize)
    n = moe.moe_forward_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    moe.moe_forward(a, ws, n)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0

    ids, w = oracle.route_topk(logits, bias, wl.k, wl.renormalize)
    ids = oracle.mark_sentinels(ids, mask, wl.E)
    assert np.array_equal(host(ids_d), ids)
    np.testing.assert_allclose(host(w_d), w, rtol=2e-6)

    g = np.random.default_rng(7)
    S = np.sort(g.choice(wl.T, 24, replace=False))
    S[0], S[-1] = 0, wl.T - 1
    S = np.unique(np.concatenate([S, np.nonzero((ids == wl.E).any(axis=1))[0][:4]]))   # tokens with sentinels
    used = np.unique(ids[S][ids[S] != wl.E])
    remap = np.full(wl.E + 1, -1, np.int64)
    remap[used] = np.arange(used.size)
    remap[wl.E] = used.size                                  # the sentinel id of the reduced layer
    ref = oracle.moe_forward(x[S], W1[used], W2[used], E=int(used.size), k=wl.k,
                             ids=remap[ids[S]].astype(np.int32), w=w[S])["out"]
    err = row_rel_err(host_f32_from_bf16(out)[S], ref)
    assert err.max() <= 2e-2, err.max()
