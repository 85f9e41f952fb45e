"""Full-size parity: every layer workload at its real size, run through
moe_forward exactly as bench.py launches it, checked against the oracle
on all routing outputs (bit-exact) and on sampled tokens (the oracle computes
those tokens one by one; a token's output depends only on its own row).  The
sample reaches every expert: each expert's first and last routed token (the
last one in the expert's last, partial tile), plus random tokens.
Also the live-row sweep of the grouped GEMMs (16384 permuted rows, 128
experts, 100 % / 50 % / 12.5 % live): sampled rows against the oracle and every
sentinel row exactly zero although its input is NaN."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_serving_gb300 import synth
from tests.gpu_helpers import (dev, dev_bf16, host, host_bf16_bits, host_f32_from_bf16,
                               require_gpu, row_rel_err)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# random tokens per workload, on top of the first and the last routed token
# of every expert (the latter lands in the expert's last, partial tile)
SAMPLE = {"32e-top4-h2880": 16, "128e-top8-h2048-zipf": 16, "256e-top8-h7168-fp8": 8,
          # decode-sized batches of the same layers (64 tokens)
          "32e-top4-h2880-t64": 16, "256e-top8-h7168-fp8-t64": 8}
CHUNK = 8                                    # experts per oracle call
THREADS = max(1, min(8, os.cpu_count() or 1))


def _sample_tokens(ids, E, k, n_random, seed):
    """Tokens that reach every expert with rows: each expert's first and last
    row in expert order (the last row sits in the expert's last tile, the
    partial one), plus n_random tokens drawn at random."""
    sr, _, off = oracle.sort_by_expert(ids, E)
    toks = set(np.random.default_rng(seed).choice(ids.shape[0], n_random, replace=False).tolist())
    for e in range(E):
        if off[e + 1] > off[e]:
            toks.add(int(sr[off[e]]) // k)
            toks.add(int(sr[off[e + 1] - 1]) // k)
    S = np.array(sorted(toks))
    assert set(np.unique(ids[S])) == set(np.nonzero(np.diff(off) > 0)[0].tolist())
    return S


def _oracle_rows(moe, wl, x, ids, w, S, W1_dev, W2_dev, S1_dev, S2_dev):
    """The oracle's layer output for tokens S, summed over chunks of CHUNK
    experts (each call sees only its chunk's experts; the other picks are
    sentinels to it -- the partial-output sum of expert parallelism), chunks in
    parallel threads.  For FP8 each chunk's weights are quantised by the
    oracle from the bf16 draws and must equal the library's, bit for bit."""
    fp8 = wl.dtype == "fp8"
    used = np.unique(ids[S])
    chunks = [used[i:i + CHUNK] for i in range(0, used.size, CHUNK)]
    xs, ids_s, w_s = x[S], ids[S], w[S]

    def run(c):
        remap = np.full(wl.E + 1, c.size, np.int64)          # other experts: sentinel of the chunk
        remap[c] = np.arange(c.size)
        W1h = synth.expert_weights(wl, "w1", experts=c, threads=2)
        W2h = synth.expert_weights(wl, "w2", experts=c, threads=2)
        kw = dict(E=int(c.size), k=wl.k, ids=remap[ids_s].astype(np.int32), w=w_s)
        if not fp8:
            return oracle.moe_forward(xs, W1h, W2h, **kw)["out"], True
        q1, s1 = oracle.quant_weight_fp8(W1h)
        q2, s2 = oracle.quant_weight_fp8(W2h)
        del W1h, W2h
        same = all(np.array_equal(host(dv[c]), hv) for dv, hv in
                   ((W1_dev, q1), (W2_dev, q2), (S1_dev, s1), (S2_dev, s2)))
        return oracle.moe_forward(xs, q1, q2, W1_scales=s1, W2_scales=s2, **kw)["out"], same

    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(run, chunks))
    assert all(same for _, same in parts), "library FP8 weight quantiser differs from the oracle's"
    return np.sum([p.astype(np.float64) for p, _ in parts], axis=0)


def _group_rel_err(y, ref, group=128):
    """Per row and 128-column group (the last one may be short):
    max |y - ref| / max |ref| over the group."""
    n = ref.shape[1]
    errs = []
    for c0 in range(0, n, group):
        errs.append(row_rel_err(y[:, c0:c0 + group], ref[:, c0:c0 + group]))
    return np.stack(errs, axis=1)


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

    # sampled tokens through the oracle: every expert's first and last row
    S = _sample_tokens(ids, wl.E, wl.k, SAMPLE[name], seed=123)
    ref = _oracle_rows(moe, wl, x, ids, w, S, W1, W2, S1, S2)
    tol = 4e-2 if fp8 else 2e-2
    got = host_f32_from_bf16(out)[S]
    err = row_rel_err(got, ref)
    assert err.max() <= tol, (name, err.max())
    # and every 128-column group on its own, the short tail group included
    # (H = 2880 = 22 * 128 + 64), against the group's own largest value
    gerr = _group_rel_err(got, ref)
    assert gerr.max() <= 2 * tol, (name, np.unravel_index(gerr.argmax(), gerr.shape), gerr.max())


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
